"""The bounded waits on the GPU: a barrier wait that nothing completes gives
up after its limit, records PA_DEVERR_TIMEOUT and returns; the context stays
usable (a decode right after it matches the oracle, the error word reads
clear again).  No fault, trap or hang is involved: the wait is bounded by
design and its limit is 50 ms here."""
import time

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


def test_an_expired_wait_is_recorded_and_the_context_stays_usable():
    from paged_kv_cache_76_gb300 import _lib, ops
    assert ops.get_device_error() == 0
    t0 = time.perf_counter()
    ops.selftest_wait_timeout(50)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.04 <= waited < 1.5, waited          # it gave up after about its limit
    assert ops.get_device_error() == _lib.PA_DEVERR_TIMEOUT
    assert ops.get_device_error() == 0           # read and cleared
    # the next work on the same context runs normally
    wl = W.custom_decode(3, 0, 0, 32, 8, 128, 16, "bf16", seed=9, split_tokens=128, lens=[300, 17, 1000])
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    torch.cuda.synchronize()
    assert_close(dev.out_decode, oracle_step(wl, vals)["decode"], "decode after an expired wait")
    assert ops.get_device_error() == 0
