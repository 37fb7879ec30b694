"""Batch-size limits on the GPU: an empty batch (and an empty prefill, copy
or scatter) is a no-op, and the largest batch the grid allows (65535
requests) decodes and verifies correctly on sampled rows, the verify on both
kernels (against the float64 oracle on a compacted copy of the blocks they
read)."""
import numpy as np
import pytest
import torch

from oracle import paged_attention as opa
from tests.paged_step import assert_close, to_f64

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


def ops():
    from paged_kv_cache_76_gb300 import ops as o
    return o


def test_empty_batch_is_a_no_op():
    kc = torch.randn(4, 16, 2, 128, device="cuda").to(torch.bfloat16)
    vc = torch.randn_like(kc)
    q = torch.empty(0, 8, 128, device="cuda", dtype=torch.bfloat16)
    tables = torch.empty(0, 2, device="cuda", dtype=torch.int32)
    lens = torch.empty(0, device="cuda", dtype=torch.int32)
    out = ops().decode(q, kc, vc, tables, lens, 0.1)
    assert out.shape == (0, 8, 128)
    q4 = torch.empty(0, 3, 8, 128, device="cuda", dtype=torch.bfloat16)
    out4 = ops().verify_decode(q4, kc, vc, tables, lens, 0.1)
    assert out4.shape == (0, 3, 8, 128)
    out5 = ops().verify_decode_tc(q4, kc, vc, tables, lens, 0.1)
    assert out5.shape == (0, 3, 8, 128)
    # no prefill request, no new token, no block pair: nothing runs, nothing is written
    kc0, vc0 = kc.clone(), vc.clone()
    qp = torch.empty(0, 8, 128, device="cuda", dtype=torch.bfloat16)
    q_start = torch.zeros(1, device="cuda", dtype=torch.int32)
    outp = ops().chunked_prefill(qp, q_start, lens, kc, vc, tables, 0.1, 0)
    assert outp.shape == (0, 8, 128)
    kn = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    ops().reshape_and_cache(kn, kn, torch.empty(0, device="cuda", dtype=torch.int32), kc, vc)
    ops().copy_blocks(kc, vc, torch.empty(0, 2, device="cuda", dtype=torch.int32))
    torch.cuda.synchronize()
    assert torch.equal(kc, kc0) and torch.equal(vc, vc0)
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("q_len,tc", [(1, False), (3, False), (3, True)], ids=["decode", "verify", "verify_tc"])
def test_the_largest_batch_matches_the_oracle_on_sampled_rows(q_len, tc):
    B, hq, hkv, d, bs = 65535, 4, 1, 64, 16
    rng = np.random.default_rng(7)
    lens = (1 + (np.arange(B) * 7919) % 31).astype(np.int32)   # 1..31 tokens: one or two blocks
    nblk = 2 * B
    perm = rng.permutation(nblk).astype(np.int32)
    tables = perm.reshape(B, 2)
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn(nblk, bs, hkv, d, generator=g, device="cuda").to(torch.float16)
    vc = torch.randn(nblk, bs, hkv, d, generator=g, device="cuda").to(torch.float16)
    q = torch.randn(B, q_len, hq, d, generator=g, device="cuda").to(torch.float16)
    scale = 1 / np.sqrt(d)
    t_dev = torch.from_numpy(tables).cuda()
    l_dev = torch.from_numpy(lens).cuda()
    if q_len == 1:
        out = ops().decode(q[:, 0].contiguous(), kc, vc, t_dev, l_dev, scale).unsqueeze(1)
    elif tc:  # one tcgen05 work unit per (request, KV head): 65535 of them
        out = ops().verify_decode_tc(q, kc, vc, t_dev, l_dev, scale)
    else:
        out = ops().verify_decode(q, kc, vc, t_dev, l_dev, scale)
    torch.cuda.synchronize()
    assert ops().get_device_error() == 0
    rows = sorted({0, 1, 2, B // 2, B - 2, B - 1} | set(rng.integers(0, B, 10).tolist()))
    # compact copy: the sampled requests' blocks, renumbered in order
    used = tables[rows].reshape(-1)
    kc_s = to_f64(kc[torch.from_numpy(used.astype(np.int64)).cuda()])
    vc_s = to_f64(vc[torch.from_numpy(used.astype(np.int64)).cuda()])
    t_s = np.arange(len(used), dtype=np.int32).reshape(len(rows), 2)
    l_s = [int(lens[r]) for r in rows]
    q_s = to_f64(q[rows])
    if q_len == 1:
        ref = opa.decode(q_s[:, 0], kc_s, vc_s, t_s, l_s, scale)[:, None]
    else:
        ref = opa.verify_decode(q_s, kc_s, vc_s, t_s, l_s, scale)
    assert_close(out[rows], ref, f"largest batch q_len {q_len}{' tensor cores' if tc else ''}")
