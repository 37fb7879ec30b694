"""ops.recording: launches marshalled once and issued again give the same
bits as the direct calls, and nothing runs while recording."""
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
    torch.cuda.init()


def test_recorded_decode_step_replays_to_the_same_bits():
    from paged_kv_cache_76_gb300 import ops
    wl = W.custom_decode(6, 0, 0, 32, 8, 128, 16, "bf16", seed=3, split_tokens=256,
                         lens=[700, 33, 1, 1500, 16, 257])
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    torch.cuda.synchronize()
    direct = dev.out_decode.clone()
    n0 = ops.launch_count()
    dev.out_decode.zero_()
    with ops.recording() as rec:
        dev.run()
    torch.cuda.synchronize()
    assert ops.launch_count() == n0  # recording launches nothing
    assert torch.count_nonzero(dev.out_decode) == 0
    assert len(rec.steps) >= 2
    for _ in range(3):
        dev.out_decode.zero_()
        rec()
        torch.cuda.synchronize()
        assert torch.equal(dev.out_decode, direct)
    assert ops.launch_count() > n0
    assert_close(dev.out_decode, oracle_step(wl, vals)["decode"], "recorded decode")
    # a recorded call that allocates its output and scratch keeps them alive
    with ops.recording() as rec2:
        o2 = ops.decode(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, dev.dec_lens, wl.scale,
                        split_tokens=dev.split_tokens)
    assert len(rec2.keep) == 2
    o2.fill_(float("nan"))
    rec2()
    torch.cuda.synchronize()
    assert torch.equal(o2, direct)
    assert ops.get_device_error() == 0


def test_recordings_do_not_nest():
    from paged_kv_cache_76_gb300 import ops
    with ops.recording():
        with pytest.raises(RuntimeError):
            with ops.recording():
                pass
    with ops.recording() as rec:  # the outer one ended cleanly
        pass
    assert rec.steps == []
