"""Preemption by swapping on the GPU ("2.1 PagedAttention" §7): the swap copy
between the device pool and a page-locked host pool is bit-exact against the
oracle's copy, and a request swapped out, overwritten and swapped back in
decodes to the same bits as before."""
import numpy as np
import pytest
import torch

from oracle import paged_attention as opa
from oracle.block_pool import SequenceManager

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


def raw(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("dt,shape", [(torch.bfloat16, (16, 8, 128)), (torch.float16, (4, 1, 64)),
                                      (torch.bfloat16, (32, 4, 128))])
def test_swap_copy_is_bit_exact_both_ways(dt, shape):
    g = torch.Generator().manual_seed(8)
    nb, ncpu = 40, 24
    gpu_k = torch.randint(-32768, 32767, (nb, *shape), generator=g, dtype=torch.int16)
    gpu_v = torch.randint(-32768, 32767, (nb, *shape), generator=g, dtype=torch.int16)
    cpu_k = torch.randint(-32768, 32767, (ncpu, *shape), generator=g, dtype=torch.int16)
    cpu_v = torch.randint(-32768, 32767, (ncpu, *shape), generator=g, dtype=torch.int16)
    gk, gv = gpu_k.view(dt).cuda(), gpu_v.view(dt).cuda()
    hk, hv = cpu_k.view(dt).pin_memory(), cpu_v.view(dt).pin_memory()
    # out: 17 GPU blocks to 17 swap blocks (pairs on the device)
    src = torch.randperm(nb, generator=g)[:17]
    dst = torch.randperm(ncpu, generator=g)[:17]
    out_pairs = torch.stack([src, dst], 1).to(torch.int32)
    rk, rv = opa.swap_blocks(gpu_k.numpy(), gpu_v.numpy(), cpu_k.numpy(), cpu_v.numpy(), out_pairs.tolist())
    ops().swap_blocks(gk, gv, hk, hv, out_pairs.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(raw(hk), rk) and np.array_equal(raw(hv), rv)
    # in: 9 swap blocks into GPU blocks (pairs in pinned host memory)
    src = torch.randperm(ncpu, generator=g)[:9]
    dst = torch.randperm(nb, generator=g)[:9]
    in_pairs = torch.stack([src, dst], 1).to(torch.int32).pin_memory()
    rk2, rv2 = opa.swap_blocks(rk, rv, gpu_k.numpy(), gpu_v.numpy(), in_pairs.tolist())
    ops().swap_blocks(hk, hv, gk, gv, in_pairs)
    torch.cuda.synchronize()
    assert np.array_equal(raw(gk), rk2) and np.array_equal(raw(gv), rv2)
    assert ops().get_device_error() == 0


def test_swap_between_two_device_pools_and_empty_pairs():
    g = torch.Generator(device="cuda").manual_seed(2)
    a = torch.randn(12, 16, 2, 128, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.zeros(5, 16, 2, 128, device="cuda", dtype=torch.bfloat16)
    pairs = torch.tensor([[11, 0], [3, 4], [0, 2]], dtype=torch.int32)
    ops().swap_blocks(a, a + 1, b, b.clone(), torch.empty(0, 2, dtype=torch.int32, device="cuda"))
    assert torch.count_nonzero(b) == 0
    bk, bv = b.clone(), b.clone()
    ops().swap_blocks(a, a + 1, bk, bv, pairs.cuda())
    for s, d in pairs.tolist():
        assert torch.equal(bk[d], a[s]) and torch.equal(bv[d], a[s] + 1)
    assert torch.count_nonzero(bk[1]) == 0 and torch.count_nonzero(bk[3]) == 0
    assert ops().get_device_error() == 0


def test_out_of_range_ids_are_recorded_and_skipped():
    from paged_kv_cache_76_gb300 import _lib
    a = torch.ones(6, 4, 1, 64, device="cuda", dtype=torch.float16)
    h = torch.zeros(3, 4, 1, 64, dtype=torch.float16).pin_memory()
    pairs = torch.tensor([[0, 3], [6, 0], [1, 1]], dtype=torch.int32, device="cuda")
    ops().swap_blocks(a, a, h, h.clone().pin_memory(), pairs)
    torch.cuda.synchronize()
    assert ops().get_device_error() == _lib.PA_DEVERR_BLOCK_ID
    assert torch.count_nonzero(h[0]) == 0 and torch.all(h[1] == 1)


def test_pageable_host_memory_is_rejected():
    from paged_kv_cache_76_gb300 import _lib
    a = torch.zeros(4, 16, 1, 64, device="cuda", dtype=torch.bfloat16)
    h = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16)              # not pinned
    pairs = torch.tensor([[0, 0]], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        ops().swap_blocks(a, a, h, h, pairs)
    st = _lib.lib().pa_swap_blocks(a.data_ptr(), a.data_ptr(), h.data_ptr(), h.data_ptr(), pairs.data_ptr(), 1,
                                   4, 4, 16, 1, 64, _lib.PA_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PA_ERR_INVALID
    assert ops().get_device_error() == 0


def test_preempted_request_decodes_to_the_same_bits_after_swap_in():
    """Allocator + kernels end to end: fill two requests, decode, swap request 0
    out, let a new request overwrite every free GPU block, swap 0 back in (into
    other physical blocks) and decode again."""
    from paged_kv_cache_76_gb300.allocator import BlockAllocator
    nb, ncpu, bs, hq, hkv, d = 64, 48, 16, 16, 4, 128
    lens = [700, 300]
    order = np.random.default_rng(0).permutation(nb).astype(np.int32)
    al, om = BlockAllocator(nb, bs, order), SequenceManager(nb, bs, order)
    for m in (al, om):
        m.enable_swap(ncpu)
    g = torch.Generator(device="cuda").manual_seed(9)
    kc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    hk = torch.zeros(ncpu, bs, hkv, d, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros(ncpu, bs, hkv, d, dtype=torch.bfloat16).pin_memory()
    for s, L in enumerate(lens):
        al.add_seq(s)
        om.add_seq(s)
        slots = al.append_slots(s, L)
        assert slots.tolist() == om.append_slots(s, L)
        k = torch.randn(L, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn(L, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
        ops().reshape_and_cache(k, v, torch.from_numpy(slots).cuda(), kc, vc)
    q = torch.randn(2, hq, d, generator=g, device="cuda").to(torch.bfloat16)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1 / np.sqrt(d)

    def decode():
        tables, _ = al.build_tables([0, 1], 64)
        return ops().decode(q, kc, vc, torch.from_numpy(tables).cuda(), lens_t, scale)

    before = decode()
    table0 = al.block_table(0)
    pairs = al.swap_out(0)
    assert pairs.tolist() == [list(p) for p in om.swap_out(0)]
    assert pairs[:, 0].tolist() == table0
    ops().swap_blocks(kc, vc, hk, hv, torch.from_numpy(pairs).cuda())
    # a new request takes every free GPU block and writes garbage into it
    al.add_seq(2)
    n_free = al.num_free()
    junk = al.append_slots(2, n_free * bs)
    ops().reshape_and_cache(torch.full((junk.size, hkv, d), 7.0, device="cuda", dtype=torch.bfloat16),
                            torch.full((junk.size, hkv, d), -7.0, device="cuda", dtype=torch.bfloat16),
                            torch.from_numpy(junk).cuda(), kc, vc)
    al.free_seq(2)
    back = al.swap_in(0)
    ops().swap_blocks(hk, hv, kc, vc, torch.from_numpy(back).pin_memory())
    new0 = al.block_table(0)
    assert new0 != table0 and back[:, 1].tolist() == new0
    after = decode()
    assert torch.equal(before, after)
    assert ops().get_device_error() == 0
