"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bit-exact for reshape_and_cache, copy_blocks and allocator indexing; attention
within max-abs 1e-2 and mean-abs 1e-3 of the oracle (bf16/fp16 in and out,
fp32 accumulation).  Bitwise equality where the method fixes it: physical
block relabelling, shared vs copied blocks, stale data past the context.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_attention as opa
from tests.paged_step import DeviceStep, assert_close, oracle_step, raw16, to_f64

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


def no_device_error():
    assert ops().get_device_error() == 0


# ---------------------------------------------------------------- tiny config
def test_tiny_config_matches_the_oracle_and_the_worked_example():
    wl = W.tiny_paged_decode()
    vals = W.make_values(wl)
    d = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    assert d.alloc.block_table(0) == [7, 2, 5] == ref["manager"].block_table(0)
    assert d.slots_host.tolist() == ref["slots"]
    d.run()
    torch.cuda.synchronize()
    assert np.array_equal(to_f64(d.k_cache), ref["k_cache"])
    assert np.array_equal(to_f64(d.v_cache), ref["v_cache"])
    assert_close(d.out_decode, ref["decode"], "tiny decode")
    no_device_error()


# ---------------------------------------------------------------- bit-exact copies
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_reshape_and_cache_is_bit_exact_on_arbitrary_bits(dt):
    g = torch.Generator().manual_seed(5)
    nb, bs, hkv, d = 40, 16, 4, 128
    pool = torch.randint(-32768, 32767, (nb, bs, hkv, d), generator=g, dtype=torch.int16)
    k = torch.randint(-32768, 32767, (300, hkv, d), generator=g, dtype=torch.int16)
    v = torch.randint(-32768, 32767, (300, hkv, d), generator=g, dtype=torch.int16)
    slots = torch.randperm(nb * bs, generator=g)[:300].to(torch.int32)
    slots[::7] = -1                                   # padding tokens
    kc, vc = pool.clone(), pool.clone()
    rk, rv = opa.reshape_and_cache(k.numpy(), v.numpy(), slots.numpy(), kc.numpy(), vc.numpy())
    dk, dv = kc.view(dt).cuda(), vc.view(dt).cuda()
    ops().reshape_and_cache(k.view(dt).cuda(), v.view(dt).cuda(), slots.cuda(), dk, dv)
    assert np.array_equal(raw16(dk), rk) and np.array_equal(raw16(dv), rv)
    no_device_error()


def test_copy_blocks_is_bit_exact():
    g = torch.Generator().manual_seed(6)
    nb, bs, hkv, d = 30, 16, 8, 128
    pool = torch.randint(-32768, 32767, (nb, bs, hkv, d), generator=g, dtype=torch.int16)
    perm = torch.randperm(nb, generator=g)
    pairs = torch.stack([perm[:10], perm[10:20]], 1).to(torch.int32)
    rk, rv = opa.copy_blocks(pool.numpy(), (pool + 1).numpy(), pairs.tolist())
    dk, dv = pool.view(torch.bfloat16).cuda(), (pool + 1).view(torch.bfloat16).cuda()
    ops().copy_blocks(dk, dv, pairs.cuda())
    assert np.array_equal(raw16(dk), rk) and np.array_equal(raw16(dv), rv)
    no_device_error()


# ---------------------------------------------------------------- decode matrix
DECODE_CASES = [
    # q_heads, kv_heads, head_dim, block_size, dtype, lens, split_tokens
    (8, 8, 128, 16, "bf16", [1, 16, 17, 100], 0),
    (2, 1, 64, 4, "fp16", [9, 5, 1, 4, 13], 0),
    (32, 8, 128, 16, "bf16", [511, 512, 513, 1000, 1537], 0),
    (28, 4, 128, 16, "bf16", [300, 1029, 2048, 17], 256),
    (64, 8, 128, 16, "bf16", [4096, 3000], 512),
    (32, 2, 128, 16, "bf16", [700, 33, 1], 0),
    (16, 4, 64, 8, "fp16", [77, 300, 8, 9], 64),
    (16, 2, 128, 32, "bf16", [33, 64, 65, 900], 128),
    (8, 4, 64, 32, "bf16", [31, 32, 1000], 0),
    (4, 4, 128, 4, "bf16", [3, 400, 1025], 256),
    (12, 3, 64, 16, "fp16", [2050, 16, 15], 1024),
    # the largest partitions (256 table entries per warp) on both block sizes
    (8, 2, 128, 16, "bf16", [4096, 4097, 9000, 1], 4096),
    (4, 1, 64, 4, "fp16", [1024, 1025, 2100], 1024),
    # 16-token partitions: exactly 32 partitions in the widest row (the
    # one-warp merge at its limit, lane c = partition c) ...
    (8, 2, 128, 16, "bf16", [512, 500, 17, 1], 16),
    (16, 4, 64, 16, "fp16", [511, 512, 33], 16),
    # ... and more than 32 (the block-per-row merge), up to 512 partitions
    (8, 2, 128, 16, "bf16", [1, 512, 513, 528, 2000], 16),
    (16, 4, 64, 16, "fp16", [2000, 512, 513, 528, 1], 16),
    (8, 8, 128, 16, "fp16", [3000, 700, 16], 16),
    (16, 4, 64, 16, "bf16", [528, 16, 4000], 16),
    (4, 1, 64, 4, "bf16", [128, 129, 700], 16),
    (16, 2, 128, 32, "bf16", [1024, 1056, 2000], 32),
    (64, 8, 128, 16, "bf16", [8192, 4097, 33], 16),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"{c[0]}q{c[1]}kv_d{c[2]}_bs{c[3]}_{c[4]}_s{c[6]}")
def test_decode_matches_the_oracle(case):
    hq, hkv, d, bs, dt, lens, split = case
    wl = W.custom_decode(len(lens), 0, 0, hq, hkv, d, bs, dt, seed=sum(lens) + hq, split_tokens=split, lens=lens)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    assert [dev.alloc.block_table(s) for s in wl.decode_seqs] == \
        [ref["manager"].block_table(s) for s in wl.decode_seqs]
    dev.run()
    torch.cuda.synchronize()
    assert np.array_equal(to_f64(dev.k_cache), ref["k_cache"])
    assert_close(dev.out_decode, ref["decode"], f"decode {case}")
    no_device_error()


def test_decode_partial_then_merge_equals_decode_and_unsplit():
    """Two launches (partial + merge) == pa_decode; split and unsplit agree within tolerance."""
    o = ops()
    wl = W.custom_decode(6, 600, 3000, 32, 8, 128, 16, "bf16", seed=3, split_tokens=256)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    a = dev.out_decode.clone()
    out = torch.empty_like(a)
    o.decode_partial(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, dev.dec_lens, wl.scale, out,
                     split_tokens=256, workspace=dev.workspace)
    o.lse_merge(dev.workspace, dev.dec_lens, dev.q_decode, dev.dec_tables, wl.block_size, out, split_tokens=256)
    assert torch.equal(out, a)
    whole = o.decode(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, dev.dec_lens, wl.scale,
                     split_tokens=4096)
    ref = oracle_step(wl, vals)["decode"]
    assert_close(whole, ref, "unsplit")
    assert_close(a, ref, "split")
    no_device_error()


# ---------------------------------------------------------------- invariants (bitwise)
def _relabelled(dev: DeviceStep, wl: W.Workload, vals, seed):
    """Same logical contents under another physical layout (free order from ``seed``)."""
    rng = np.random.default_rng(seed)
    wl2 = W.Workload(**{**wl.__dict__, "free_order": rng.permutation(wl.num_blocks).astype(np.int32)})
    dev2 = DeviceStep(wl2, vals)
    # pool2[table2[r][j]] = pool1[table1[r][j]] for every used logical block; every other block NaN
    k2 = torch.full_like(dev.k_cache, float("nan"))
    v2 = torch.full_like(dev.v_cache, float("nan"))
    seqs = sorted(wl.decode_seqs + [s for s, _, _ in wl.prefill])
    src, dst = [], []
    for s in seqs:
        src += dev.alloc.block_table(s)
        dst += dev2.alloc.block_table(s)
    src = torch.as_tensor(src, device="cuda")
    dst = torch.as_tensor(dst, device="cuda")
    pre_k, pre_v = vals["k_cache"].cuda(), vals["v_cache"].cuda()
    k2[dst] = pre_k[src]
    v2[dst] = pre_v[src]
    dev2.k_cache, dev2.v_cache = k2, v2
    return dev2


@pytest.mark.parametrize("split", [0, 128])
def test_physical_relabelling_gives_bitwise_identical_output(split):
    wl = W.custom_decode(12, 1, 1500, 32, 8, 128, 16, "bf16", seed=11, split_tokens=split)
    vals = W.make_values(wl)
    a = DeviceStep(wl, vals)
    b = _relabelled(a, wl, vals, seed=99)
    a.run()
    b.run()
    assert torch.equal(a.out_decode, b.out_decode)
    no_device_error()


def test_identity_table_equals_a_contiguous_layout():
    o = ops()
    lens = [37, 512, 1000, 16]
    hq, hkv, d, bs = 16, 4, 128, 16
    nblk = [-(-L // bs) for L in lens]
    nb = sum(nblk)
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(len(lens), hq, d, generator=g, device="cuda").to(torch.bfloat16)
    ident = torch.full((len(lens), max(nblk)), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(nblk):
        ident[r, :n] = torch.arange(off, off + n)
        off += n
    ident = ident.cuda()
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out_id = o.decode(q, kc, vc, ident, lens_t, 1 / np.sqrt(d))
    # contiguous attention per request (oracle on the identity layout) ...
    ref = opa.decode(to_f64(q), to_f64(kc), to_f64(vc), ident.cpu().numpy(), lens, 1 / np.sqrt(d))
    assert_close(out_id, ref, "identity")
    # ... and a random relabelling of the same blocks gives the same bits
    pi = torch.randperm(nb, generator=torch.Generator().manual_seed(4)).cuda()
    k2, v2 = torch.empty_like(kc), torch.empty_like(vc)
    k2[pi] = kc
    v2[pi] = vc
    t2 = torch.where(ident >= 0, pi[ident.clamp(min=0).long()].int(), ident)
    out2 = o.decode(q, k2, v2, t2, lens_t, 1 / np.sqrt(d))
    assert torch.equal(out_id, out2)
    no_device_error()


def test_stale_and_freed_data_past_the_context_is_invisible():
    """A freed request's blocks are reused without clearing; NaN/huge stale values change nothing."""
    wl = W.custom_decode(4, 0, 0, 16, 4, 128, 16, "bf16", seed=21, lens=[150, 200, 37, 90], pool_factor=4.0)
    wl.setup_ops = [("add", 100), ("append", 100, 333), ("free", 100)] + wl.setup_ops
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    clean = dev.out_decode.clone()
    # poison every slot not inside a live context (after this step's writes)
    live = torch.zeros(wl.num_blocks * wl.block_size, dtype=torch.bool)
    for s, L in zip(wl.decode_seqs, dev.dec_lens_host):
        t = dev.alloc.block_table(s)
        for pos in range(int(L)):
            live[t[pos // wl.block_size] * wl.block_size + pos % wl.block_size] = True
    dead = (~live).cuda().view(wl.num_blocks, wl.block_size)
    for poison in (float("nan"), 3.0e38):
        vals2 = dict(vals)
        kc, vc = vals["k_cache"].cuda().clone(), vals["v_cache"].cuda().clone()
        kc[dead] = poison
        vc[dead] = poison
        vals2["k_cache"], vals2["v_cache"] = kc, vc
        d2 = DeviceStep(wl, vals2)
        d2.run()
        assert torch.equal(d2.out_decode, clean)
    assert_close(clean, oracle_step(wl, vals)["decode"], "stale")
    no_device_error()


def test_zero_context_gives_a_zero_row():
    wl = W.custom_decode(3, 5, 40, 8, 2, 128, 16, "bf16", seed=4)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    lens = dev.dec_lens.clone()
    lens[1] = 0
    out = ops().decode(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, lens, wl.scale)
    assert torch.count_nonzero(out[1]) == 0
    assert torch.equal(out[0], dev.out_decode[0]) and torch.equal(out[2], dev.out_decode[2])
    no_device_error()


# ---------------------------------------------------------------- sharing and copy-on-write
def test_prefix_sharing_and_cow_give_identical_results():
    wl = W.prefix_shared_cow_decode(batch=24, prefix_tokens=512, suffix_lo=16, suffix_hi=200, cow_frac=0.25)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    assert len(dev.pairs_host) == 6 and dev.pairs_host.tolist() == [list(p) for p in ref["pairs"]]
    dev.run()
    assert_close(dev.out_decode, ref["decode"], "prefix+cow")
    # the same step without the copy-on-write: identical outputs, bit for bit
    wl_nocow = W.Workload(**{**wl.__dict__, "step_ops": [op for op in wl.step_ops if op[0] != "cow"]})
    dev2 = DeviceStep(wl_nocow, vals)
    dev2.run()
    assert torch.equal(dev.out_decode, dev2.out_decode)
    no_device_error()


def test_copy_on_write_of_a_partial_shared_block():
    """Writer copies the half-full shared block and appends into the copy; sharers are unaffected."""
    bs, holder = 16, 50
    wl = W.custom_decode(4, 0, 0, 32, 8, 128, bs, "bf16", seed=8, lens=[1, 1, 1, 1])
    wl.num_blocks = 40
    wl.free_order = np.random.default_rng(8).permutation(40).astype(np.int32)
    wl.setup_ops = [("add", holder), ("append", holder, 40)]   # blocks: 16 + 16 + 8 tokens
    for s in range(4):
        wl.setup_ops += [("add", s), ("share", s, holder, 40)]
    wl.setup_ops += [("free", holder)]                         # refcounts now 4
    wl.step_ops = [("cow", 0, 2), ("append", 0, 8)]            # seq 0 diverges inside block 2
    wl.decode_lens = [48, 40, 40, 40]
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    assert dev.pairs_host.tolist() == [list(p) for p in ref["pairs"]] and len(ref["pairs"]) == 1
    src = int(dev.pairs_host[0, 0])
    assert dev.alloc.ref(src) == 3
    before = vals["k_cache"][src].clone()
    dev.run()
    assert_close(dev.out_decode, ref["decode"], "partial cow")
    assert torch.equal(dev.k_cache[src].cpu(), before)            # the shared original is untouched
    # the sharers see exactly what they saw before anyone wrote
    wl_ro = W.Workload(**{**wl.__dict__, "step_ops": [], "decode_lens": [40, 40, 40, 40]})
    dev_ro = DeviceStep(wl_ro, {**vals, "k_new": vals["k_new"][:0], "v_new": vals["v_new"][:0]})
    dev_ro.run()
    assert torch.equal(dev.out_decode[1:], dev_ro.out_decode[1:])
    no_device_error()


# ---------------------------------------------------------------- chunked prefill
PREFILL_CASES = [
    # q_heads, kv_heads, head_dim, block_size, dtype, histories, chunks
    (28, 4, 128, 16, "bf16", [0, 5, 300], [64, 17, 100]),
    (8, 8, 128, 16, "bf16", [1000, 0], [1, 129]),
    (4, 1, 64, 4, "fp16", [7, 33], [9, 40]),
    (16, 2, 128, 32, "bf16", [64, 65], [63, 70]),
    (32, 2, 64, 8, "fp16", [130, 0], [31, 256]),
    # a request with an empty chunk between two others, on both prefill kernels
    (8, 2, 128, 16, "bf16", [100, 40, 0], [33, 0, 20]),
    (4, 1, 64, 4, "fp16", [7, 0, 12], [0, 9, 5]),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: f"{c[0]}q{c[1]}kv_d{c[2]}_bs{c[3]}_{c[4]}")
def test_chunked_prefill_matches_the_oracle(case):
    hq, hkv, d, bs, dt, hists, chunks = case
    rng = np.random.default_rng(hq + d)
    needed = sum(-(-(h + c) // bs) for h, c in zip(hists, chunks)) + 4
    nb = int(1.5 * needed)
    setup, step, prefill = [], [], []
    for i, (h, c) in enumerate(zip(hists, chunks)):
        setup.append(("add", i))
        if h:
            setup.append(("append", i, h))
        step.append(("append", i, c))
        prefill.append((i, c, h + c))
    wl = W.Workload(name="prefill_case", dtype=dt, q_heads=hq, kv_heads=hkv, head_dim=d, block_size=bs,
                    num_blocks=nb, scale=1.0 / np.sqrt(d), free_order=rng.permutation(nb).astype(np.int32),
                    setup_ops=setup, step_ops=step, prefill=prefill, seed=hq)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    dev.run()
    assert np.array_equal(to_f64(dev.k_cache), ref["k_cache"])
    assert_close(dev.out_prefill, ref["prefill"], f"prefill {case}")
    no_device_error()


@pytest.mark.parametrize("max_ctas", [1, 2, 3, 7])
def test_chunked_prefill_with_few_ctas_matches_one_cta_per_unit(max_ctas):
    """The tensor-core path with max_ctas CTAs looping over work units (each
    CTA carries its barrier phases and TMEM across several units, some of them
    empty) gives bit-identical output to one CTA per unit, and matches the
    oracle."""
    o = ops()
    hq, hkv, d, bs = 16, 2, 128, 16
    hists, chunks = [300, 0, 41, 1000], [97, 200, 16, 130]
    rng = np.random.default_rng(5)
    needed = sum(-(-(h + c) // bs) for h, c in zip(hists, chunks)) + 4
    nb = int(1.5 * needed)
    setup, step, prefill = [], [], []
    for i, (h, c) in enumerate(zip(hists, chunks)):
        setup.append(("add", i))
        if h:
            setup.append(("append", i, h))
        step.append(("append", i, c))
        prefill.append((i, c, h + c))
    wl = W.Workload(name="prefill_few_ctas", dtype="bf16", q_heads=hq, kv_heads=hkv, head_dim=d, block_size=bs,
                    num_blocks=nb, scale=1.0 / np.sqrt(d), free_order=rng.permutation(nb).astype(np.int32),
                    setup_ops=setup, step_ops=step, prefill=prefill, seed=11)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    dev.run()
    no_device_error()
    full = dev.out_prefill.clone()
    out = torch.full_like(full, float("nan"))
    o.chunked_prefill(dev.q_prefill, dev.q_start, dev.pre_lens, dev.k_cache, dev.v_cache, dev.pre_tables,
                      wl.scale, dev.max_q_len, out=out, max_ctas=max_ctas)
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(out, full)
    assert_close(out, ref["prefill"], f"prefill max_ctas={max_ctas}")


def test_mixed_prefill_and_decode_step():
    wl = W.mixed_prefill_decode(n_prefill=2, chunk=128, hist_lo=0, hist_hi=700, n_decode=12, dec_lo=256,
                                dec_hi=2000)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    ref = oracle_step(wl, vals)
    dev.run()
    assert np.array_equal(to_f64(dev.k_cache), ref["k_cache"])
    assert_close(dev.out_prefill, ref["prefill"], "mixed prefill")
    assert_close(dev.out_decode, ref["decode"], "mixed decode")
    no_device_error()


# ---------------------------------------------------------------- device-side checks
def test_bad_indices_are_recorded_not_faulted():
    from paged_kv_cache_76_gb300 import _lib
    o = ops()
    wl = W.custom_decode(3, 40, 90, 8, 2, 128, 16, "bf16", seed=2)
    vals = W.make_values(wl)
    dev = DeviceStep(wl, vals)
    dev.run()
    no_device_error()
    good = dev.out_decode.clone()
    # a block id past the pool in request 1's table
    tables = dev.dec_tables.clone()
    tables[1, 0] = wl.num_blocks + 5
    out = o.decode(dev.q_decode, dev.k_cache, dev.v_cache, tables, dev.dec_lens, wl.scale)
    assert o.get_device_error() == _lib.PA_DEVERR_BLOCK_ID
    assert torch.equal(out[0], good[0]) and torch.equal(out[2], good[2])
    assert o.get_device_error() == 0                         # reading clears it
    # a context longer than the table
    lens = dev.dec_lens.clone()
    longest = int(torch.argmax(lens))                        # its table row is full: no bad ids read
    lens[longest] = tables.shape[1] * wl.block_size + 1
    o.decode(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, lens, wl.scale)
    assert o.get_device_error() == _lib.PA_DEVERR_CONTEXT_LEN
    # a slot past the pool: recorded, the other tokens still land
    slots = dev.slots.clone()
    slots[0] = wl.num_blocks * wl.block_size
    o.reshape_and_cache(dev.k_new, dev.v_new, slots, dev.k_cache, dev.v_cache)
    assert o.get_device_error() == _lib.PA_DEVERR_SLOT
    # a copy pair out of range
    o.copy_blocks(dev.k_cache, dev.v_cache, torch.tensor([[0, wl.num_blocks]], dtype=torch.int32, device="cuda"))
    assert o.get_device_error() == _lib.PA_DEVERR_BLOCK_ID
    # a prefill chunk longer than the declared maximum
    qs = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    o.chunked_prefill(dev.q_decode[:1].expand(8, -1, -1).contiguous(), qs, dev.dec_lens[:1], dev.k_cache,
                      dev.v_cache, dev.dec_tables[:1], wl.scale, max_q_len=4)
    assert o.get_device_error() == _lib.PA_DEVERR_QUERY_RANGE
    # the context is still healthy
    dev.run()
    assert torch.equal(dev.out_decode, good)
    no_device_error()


def test_launch_counter_counts_kernels():
    o = ops()
    wl = W.custom_decode(2, 600, 900, 8, 2, 128, 16, "bf16", seed=1)
    dev = DeviceStep(wl, W.make_values(wl))
    n0 = o.launch_count()
    dev.run()                 # reshape_and_cache + decode partial + merge
    assert o.launch_count() - n0 == 3
