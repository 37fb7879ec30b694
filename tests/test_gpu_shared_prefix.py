"""GPU parity of pa_decode_shared_prefix (shared prefix on the tensor cores +
per-request suffix decode + log-sum-exp merge) against the float64 oracle and
against pa_decode on the full tables."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.paged_step import DeviceStep, assert_close, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_76_gb300 import _lib
    try:
        _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()


def _shared(dev: DeviceStep):
    """The blocks every decode request shares, from the C++ allocator."""
    nblk = dev.alloc.common_prefix(dev.wl.decode_seqs)
    blocks = dev.alloc.block_table(dev.wl.decode_seqs[0])[:nblk]
    return torch.tensor(blocks, dtype=torch.int32, device="cuda"), nblk * dev.wl.block_size


def _run(dev):
    from paged_kv_cache_76_gb300 import ops
    dev.run()  # copy_blocks + reshape_and_cache + pa_decode on the full tables
    pb, plen = _shared(dev)
    out = ops.decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache, pb, plen, dev.dec_tables, dev.dec_lens,
                                   dev.wl.scale)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    return out, plen


@pytest.mark.parametrize("hq,hkv,d,bs,dt", [(32, 8, 128, 16, "bf16"), (16, 2, 64, 8, "fp16"), (28, 4, 128, 32, "bf16")])
def test_shared_prefix_decode_matches_oracle_and_decode(hq, hkv, d, bs, dt):
    wl = W.prefix_shared_cow_decode(batch=24, prefix_tokens=bs * 40, suffix_lo=1, suffix_hi=300, cow_frac=0.25,
                                    q_heads=hq, kv_heads=hkv, head_dim=d, block_size=bs)
    wl.dtype = dt
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    out, plen = _run(dev)
    assert plen == bs * 39          # the copied last prefix block is private to the CoW requests
    ref = oracle_step(wl, vals)["decode"]
    assert_close(out, ref, "shared prefix")
    assert_close(dev.out_decode, ref, "plain decode")


def test_empty_and_long_suffixes():
    bs, holder = 16, 99
    wl = W.custom_decode(4, 0, 0, 32, 8, 128, bs, "bf16", seed=5, lens=[1, 1, 1, 1], pool_factor=1.0)
    wl.num_blocks = 200
    wl.free_order = np.random.default_rng(5).permutation(200).astype(np.int32)
    wl.setup_ops = [("add", holder), ("append", holder, 700)]
    for s in range(4):
        wl.setup_ops += [("add", s), ("share", s, holder, 688)]   # 43 full blocks
    wl.setup_ops += [("free", holder), ("append", 1, 4), ("append", 2, 900), ("append", 3, 15)]
    wl.step_ops = [("append", 1, 1), ("append", 2, 1), ("append", 3, 1)]
    wl.decode_lens = [688, 693, 1589, 704]
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    out, plen = _run(dev)
    assert plen == 688               # request 0 is exactly the prefix: empty suffix
    assert_close(out, oracle_step(wl, vals)["decode"], "empty/long suffix")


def test_prefix_mismatch_and_short_context_are_recorded():
    from paged_kv_cache_76_gb300 import _lib, ops
    wl = W.prefix_shared_cow_decode(batch=8, prefix_tokens=256, suffix_lo=10, suffix_hi=40, cow_frac=0.0)
    dev = DeviceStep(wl, W.make_values(wl))
    dev.run()
    pb, plen = _shared(dev)
    bad = pb.clone()
    bad[3] = (bad[3] + 1) % wl.num_blocks
    ops.decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache, bad, plen, dev.dec_tables, dev.dec_lens,
                             wl.scale)
    assert ops.get_device_error() == _lib.PA_DEVERR_BLOCK_ID
    lens = dev.dec_lens.clone()
    lens[2] = plen - 1
    ops.decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache, pb, plen, dev.dec_tables, lens, wl.scale)
    assert ops.get_device_error() == _lib.PA_DEVERR_CONTEXT_LEN
    out = ops.decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache, pb, plen, dev.dec_tables, dev.dec_lens,
                                   wl.scale)
    assert ops.get_device_error() == 0
    assert_close(out, oracle_step(wl, W.make_values(wl))["decode"], "after errors")


def test_four_token_blocks_fall_back_to_decode():
    from paged_kv_cache_76_gb300 import ops
    wl = W.prefix_shared_cow_decode(batch=6, prefix_tokens=64, suffix_lo=1, suffix_hi=30, cow_frac=0.0,
                                    q_heads=8, kv_heads=2, head_dim=64, block_size=4)
    dev = DeviceStep(wl, W.make_values(wl))
    out, _ = _run(dev)
    assert torch.equal(out, dev.out_decode)


def _concurrent(dev, pb, plen):
    """The prefix pass on a second stream forked from the current one (the
    caller's ordering duty: q and the prefix K/V are written before the fork)."""
    from paged_kv_cache_76_gb300 import ops
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=torch.cuda.Stream.priority_range()[1])
    side.wait_stream(main)
    out = ops.decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache, pb, plen, dev.dec_tables, dev.dec_lens,
                                   dev.wl.scale, prefix_stream=side)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    return out


def test_concurrent_prefix_pass_with_the_same_key_ranges_is_bitwise_the_same():
    # 24 requests x 4 heads: one pair of row tiles per KV head, so 512-token
    # ranges already fit in half of the SMs and the partials are the same
    wl = W.prefix_shared_cow_decode(batch=24, prefix_tokens=16 * 64, suffix_lo=1, suffix_hi=300, cow_frac=0.25)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    out, plen = _run(dev)
    pb, _ = _shared(dev)
    assert torch.equal(_concurrent(dev, pb, plen), out)


def test_concurrent_prefix_pass_at_full_size_matches_the_oracle():
    wl = W.prefix_shared_cow_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    pb, plen = _shared(dev)
    out = _concurrent(dev, pb, plen)
    rows = list(range(0, 256, 16))
    ref = oracle_step(wl, vals, decode_rows=rows, compact=True)["decode"]
    assert_close(out[rows], ref, "concurrent shared prefix")
    # every row against pa_decode on the full tables (two bf16 roundings apart)
    assert float(np.abs(to_f64(out) - to_f64(dev.out_decode)).mean()) < 1e-3
