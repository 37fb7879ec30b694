"""The vAttention-style comparison baseline on the GPU ("vAttention 完全拆解"):
decode over contiguous per-slot KV (plain memory and CUDA-VMM pages mapped on
demand) against the oracle and, bit for bit, against the paged kernel on the
same K/V."""
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


def va():
    from paged_kv_cache_76_gb300 import vattention
    return vattention


def ops():
    from paged_kv_cache_76_gb300 import ops as o
    return o


def _identity_tables(slot_ids, L):
    nb = L // 16
    return torch.stack([torch.arange(nb, dtype=torch.int32) + s * nb for s in slot_ids.tolist()]).cuda()


@pytest.mark.parametrize("hq,hkv,d,dt,split", [(32, 8, 128, torch.bfloat16, 0), (16, 2, 64, torch.float16, 128),
                                                (8, 8, 128, torch.bfloat16, 256)])
def test_contiguous_decode_matches_the_oracle_and_the_paged_kernel_bitwise(hq, hkv, d, dt, split):
    g = torch.Generator(device="cuda").manual_seed(1)
    S, L = 6, 1024
    kc = torch.randn(S, L, hkv, d, generator=g, device="cuda").to(dt)
    vc = torch.randn(S, L, hkv, d, generator=g, device="cuda").to(dt)
    slot_ids = torch.tensor([4, 0, 5, 2, 1], dtype=torch.int32, device="cuda")
    lens = torch.tensor([1024, 1, 17, 1000, 512], dtype=torch.int32, device="cuda")
    q = torch.randn(5, hq, d, generator=g, device="cuda").to(dt)
    scale = 1 / np.sqrt(d)
    out = va().decode_contiguous(q, kc, vc, slot_ids, lens, scale, split_tokens=split)
    # the same K/V seen as a paged pool of 16-token blocks with identity tables
    pool_k = kc.view(S * L // 16, 16, hkv, d)
    pool_v = vc.view(S * L // 16, 16, hkv, d)
    tables = _identity_tables(slot_ids.cpu(), L)
    paged = ops().decode(q, pool_k, pool_v, tables, lens, scale, split_tokens=split)
    assert torch.equal(out, paged)
    ref = opa.decode(to_f64(q), to_f64(pool_k), to_f64(pool_v), tables.cpu().numpy(), lens.tolist(), scale)
    assert_close(out, ref, "contiguous decode")
    assert ops().get_device_error() == 0


def test_slot_bounds_are_enforced_without_touching_rows_past_them():
    from paged_kv_cache_76_gb300 import _lib
    g = torch.Generator(device="cuda").manual_seed(2)
    S, L, hkv, d = 3, 256, 2, 64
    kc = torch.randn(S, L, hkv, d, generator=g, device="cuda").to(torch.float16)
    vc = torch.randn(S, L, hkv, d, generator=g, device="cuda").to(torch.float16)
    q = torch.randn(2, 4, d, generator=g, device="cuda").to(torch.float16)
    bounds = torch.tensor([64, 256, 0], dtype=torch.int32, device="cuda")
    slot_ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    lens = torch.tensor([64, 200], dtype=torch.int32, device="cuda")
    a = va().decode_contiguous(q, kc, vc, slot_ids, lens, 0.125, slot_tokens=bounds)
    assert ops().get_device_error() == 0
    # poison what lies past slot 0's bound: nothing changes
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[0, 64:] = float("nan")
    vc2[0, 64:] = float("nan")
    b = va().decode_contiguous(q, kc2, vc2, slot_ids, lens, 0.125, slot_tokens=bounds)
    assert torch.equal(a, b)
    # a context past the bound is an error, and the rows past it count as absent
    c = va().decode_contiguous(q, kc2, vc2, slot_ids, torch.tensor([100, 200], dtype=torch.int32, device="cuda"),
                               0.125, slot_tokens=bounds)
    assert ops().get_device_error() == _lib.PA_DEVERR_CONTEXT_LEN
    assert torch.equal(c, a) and torch.isfinite(c.float()).all()
    # a bad slot id: error and a zero row
    z = va().decode_contiguous(q, kc, vc, torch.tensor([7, 1], dtype=torch.int32, device="cuda"), lens, 0.125,
                               slot_tokens=bounds)
    assert ops().get_device_error() == _lib.PA_DEVERR_BLOCK_ID
    assert torch.count_nonzero(z[0]) == 0 and torch.equal(z[1], a[1])
    # writes past a bound are refused and recorded
    k1 = torch.ones(2, hkv, d, device="cuda", dtype=torch.float16)
    va().reshape_and_cache_slots(k1, k1, torch.tensor([2, 0], dtype=torch.int32, device="cuda"),
                                 torch.tensor([0, 63], dtype=torch.int32, device="cuda"), kc, vc, slot_tokens=bounds)
    assert ops().get_device_error() == _lib.PA_DEVERR_SLOT
    assert torch.all(kc[0, 63] == 1) and not torch.all(kc[2, 0] == 1)


def test_vmm_pages_map_on_demand_and_decode_equals_the_paged_kernel():
    """Slots of 2 pages each (2 MiB pages, 2 KB rows -> 1024 tokens a page):
    lengths around the page boundary, growth by steps, a finished slot reused
    with its pages, and decode against the paged kernel on the same K/V."""
    V = va()
    G = V.VirtualKV.granularity()
    hkv, d = 8, 128
    row = hkv * d * 2
    L = 2 * G // row
    S = 6
    vkv = V.VirtualKV(S, L, 1, hkv, d, torch.bfloat16, page_bytes=G, max_pages=16)
    slots = [vkv.alloc_slot() for _ in range(5)]
    assert slots == [0, 1, 2, 3, 4]
    per_page = G // row
    lens = [per_page - 1, per_page, per_page + 1, 1, 2 * per_page]
    full = np.zeros(S, dtype=np.int32)
    full[slots] = lens
    vkv.step(full)
    assert [vkv.slot_pages(s) for s in slots] == [1, 1, 2, 1, 2]
    st = vkv.stats()
    assert st["pages_mapped"] == 2 * 7 and st["map_calls"] == 14
    g = torch.Generator(device="cuda").manual_seed(3)
    kref = torch.zeros(S, L, hkv, d, dtype=torch.bfloat16, device="cuda")
    vref = torch.zeros_like(kref)
    sid, pos = [], []
    for s, n in zip(slots, lens):
        sid += [s] * n
        pos += list(range(n))
    k = torch.randn(len(sid), hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(len(sid), hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    sid_t = torch.tensor(sid, dtype=torch.int32, device="cuda")
    pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
    vkv.reshape_and_cache(0, k, v, sid_t, pos_t)
    kref[sid_t.long(), pos_t.long()] = k
    vref[sid_t.long(), pos_t.long()] = v
    assert ops().get_device_error() == 0
    q = torch.randn(5, 32, d, generator=g, device="cuda").to(torch.bfloat16)
    slot_ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = vkv.decode(0, q, slot_ids, lens_t, 1 / np.sqrt(d))
    tables = _identity_tables(slot_ids.cpu(), L)
    paged = ops().decode(q, kref.view(-1, 16, hkv, d), vref.view(-1, 16, hkv, d), tables, lens_t, 1 / np.sqrt(d))
    assert torch.equal(out, paged)
    assert ops().get_device_error() == 0
    # the virtual tensor as a torch view: only rows inside mapped pages are read
    kv0 = vkv.tensor(0, False)
    assert torch.equal(kv0[2, :1025], kref[2, :1025]) and torch.equal(kv0[4, :2048], kref[4, :2048])
    # slot 1 finishes; the next request takes the slot with the most pages among the free ones
    vkv.free_slot(1)
    full[1] = 0
    vkv.step(full)
    assert vkv.alloc_slot() == 1 and vkv.slot_pages(1) == 1
    # growth past the budget reclaims nothing active and fails cleanly
    big = full.copy()
    big[slots] = L
    with pytest.raises(V.NoPages):
        vkv.step(big)
    assert vkv.stats()["pages_mapped"] == 14
    out2 = vkv.decode(0, q, slot_ids, lens_t, 1 / np.sqrt(d))
    assert torch.equal(out2, out)
    vkv.close()
