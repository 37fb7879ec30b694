"""Automatic prefix caching end to end on the GPU ("Khám phá vLLM … phần 2",
prefix caching): a request whose prompt starts with a cached prefix prefills
only its uncached tokens over the cached blocks, and gets the attention the
full recomputation gets."""
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


@pytest.mark.parametrize("bs,hq,hkv,d", [(16, 32, 8, 128), (32, 8, 2, 64)])
def test_cache_hit_prefill_and_decode_match_the_recomputed_request(bs, hq, hkv, d):
    from paged_kv_cache_76_gb300.allocator import BlockAllocator
    nb = 256
    rng = np.random.default_rng(5)
    prefix = rng.integers(0, 1000, 300).tolist()
    tail_a, tail_b = rng.integers(0, 1000, 40).tolist(), rng.integers(0, 1000, 57).tolist()
    prompt_a, prompt_b = prefix + tail_a, prefix + tail_b
    nb_hit = len(prefix) // bs
    g = torch.Generator(device="cuda").manual_seed(6)
    # K/V of every position of either prompt: the shared prefix has the same
    # K/V in both (it depends on the tokens before it only)
    kp = torch.randn(len(prefix), hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    vp = torch.randn(len(prefix), hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    kv_tail = {n: (torch.randn(n, hkv, d, generator=g, device="cuda").to(torch.bfloat16),
                   torch.randn(n, hkv, d, generator=g, device="cuda").to(torch.bfloat16))
               for n in (len(tail_a), len(tail_b))}
    kb = torch.cat([kp, kv_tail[len(tail_b)][0]])
    vb = torch.cat([vp, kv_tail[len(tail_b)][1]])
    q_b = torch.randn(len(prompt_b), hq, d, generator=g, device="cuda").to(torch.bfloat16)
    scale = 1 / np.sqrt(d)
    kc = torch.zeros(nb, bs, hkv, d, device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)

    al = BlockAllocator(nb, bs)
    al.enable_prefix_caching()
    # request A fills (and registers) the prefix blocks, then finishes
    assert al.add_seq_cached(0, prompt_a) == 0
    slots_a = al.append_tokens(0, prompt_a)
    ka = torch.cat([kp, kv_tail[len(tail_a)][0]])
    va = torch.cat([vp, kv_tail[len(tail_a)][1]])
    ops().reshape_and_cache(ka, va, torch.from_numpy(slots_a).cuda(), kc, vc)
    al.free_seq(0)
    # request B: the prefix's full blocks hit; only the rest is written and prefilled
    hit = al.add_seq_cached(1, prompt_b)
    assert hit == nb_hit * bs
    slots_b = al.append_tokens(1, prompt_b[hit:])
    ops().reshape_and_cache(kb[hit:], vb[hit:], torch.from_numpy(slots_b).cuda(), kc, vc)
    # request C: the same prompt with nothing cached (a second allocator over the same pool ids
    # would alias; use fresh caches instead)
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    al2 = BlockAllocator(nb, bs)
    al2.add_seq(2)
    slots_c = al2.append_slots(2, len(prompt_b))
    ops().reshape_and_cache(kb, vb, torch.from_numpy(slots_c).cuda(), kc2, vc2)

    L = len(prompt_b)
    maxblk = -(-L // bs)
    t_b = torch.tensor([al.block_table(1)], dtype=torch.int32, device="cuda")
    t_c = torch.tensor([al2.block_table(2)], dtype=torch.int32, device="cuda")
    assert t_b.shape[1] == t_c.shape[1] == maxblk
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    rows = L - hit
    out_b = ops().chunked_prefill(q_b[hit:].contiguous(), torch.tensor([0, rows], dtype=torch.int32, device="cuda"),
                                  lens, kc, vc, t_b, scale, rows)
    out_c = ops().chunked_prefill(q_b, torch.tensor([0, L], dtype=torch.int32, device="cuda"), lens, kc2, vc2, t_c,
                                  scale, L)
    ref = opa.chunked_prefill(to_f64(q_b[hit:]), [0, rows], [L], to_f64(kc), to_f64(vc), t_b.cpu().numpy(), scale)
    assert_close(out_b, ref, "cache-hit prefill")
    assert_close(out_c[hit:], ref, "recomputed prefill")
    # one decode step of B against the recomputed C: same K/V bits in other blocks
    q1 = torch.randn(1, hq, d, generator=g, device="cuda").to(torch.bfloat16)
    dec_b = ops().decode(q1, kc, vc, t_b, lens, scale)
    dec_c = ops().decode(q1, kc2, vc2, t_c, lens, scale)
    assert torch.equal(dec_b, dec_c)
    assert ops().get_device_error() == 0
