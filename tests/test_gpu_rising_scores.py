"""Scores that keep rising along the context, on every attention kernel.

K is scaled by 1 + 0.35 j in the j-th block of each request's context, so a
row's maximum score grows by more than 2^8 (in base-2 units) from one
128-key tile to the next: the running maximum that the kernels keep is raised
on almost every tile and the accumulated output is rescaled each time ("Khám
phá vLLM … phần 2", the online softmax of paged attention; the result is the
plain softmax, whatever the order of the keys).  Random N(0, 1) inputs never
raise it after the first tile, so this is the case that exercises the
rescale path and its ordering against the next P.V product."""
import numpy as np
import pytest
import torch

from oracle import paged_attention as opa
from tests.paged_step import assert_close, to_f64

pytestmark = pytest.mark.gpu

GROW = 0.35


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


def _pool(seed, lens, hkv, d, bs, dt, shared_blocks=0):
    """Paged K/V for requests of ``lens`` tokens in shuffled blocks; the first
    ``shared_blocks`` blocks of every table are the same physical blocks.  K of
    a request's j-th block is scaled by 1 + GROW * j."""
    rng = np.random.default_rng(seed)
    own = [max(-(-L // bs), 1) - shared_blocks for L in lens]
    maxblk = shared_blocks + max(own) + 2
    nb = shared_blocks + sum(own) + 5
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), maxblk), -1, dtype=np.int32)
    tables[:, :shared_blocks] = perm[:shared_blocks]
    off = shared_blocks
    for r, n in enumerate(own):
        tables[r, shared_blocks:shared_blocks + n] = perm[off:off + n]
        off += n
    g = torch.Generator(device="cuda").manual_seed(seed)
    dtype = torch.bfloat16 if dt == "bf16" else torch.float16
    kc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda")
    vc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(dtype)
    grow = torch.ones(nb, device="cuda")
    for r in range(len(lens)):
        for j in range(maxblk):
            if tables[r, j] >= 0:
                grow[int(tables[r, j])] = 1.0 + GROW * j
    kc = (kc * grow[:, None, None, None]).to(dtype)
    return kc, vc, tables, g, dtype


def _check(out, ref, what):
    # a nearly one-hot softmax makes the output a V row of magnitude up to
    # ~4.5, whose own rounding to bf16 is up to 2^-8 of it (0.018): the
    # bound admits that rounding on top of 1e-2
    torch.cuda.synchronize()
    assert_close(out, ref, what, rounding=True)
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("split", [0, 256])
def test_decode(split):
    lens, hq, hkv, d, bs = [1500, 37, 700, 4000], 32, 8, 128, 16
    kc, vc, tables, g, dtype = _pool(21, lens, hkv, d, bs, "bf16")
    q = torch.randn(len(lens), hq, d, generator=g, device="cuda").to(dtype)
    scale = 1 / np.sqrt(d)
    out = ops().decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.tensor(lens, dtype=torch.int32,
                       device="cuda"), scale, split_tokens=split)
    _check(out, opa.decode(to_f64(q), to_f64(kc), to_f64(vc), tables, lens, scale), f"decode split {split}")


VERIFY_TC = [
    # q_len, q_heads, kv_heads, head_dim, block_size, dtype, lens
    (8, 32, 8, 128, 16, "bf16", [2339, 130, 17, 1500]),   # 32 rows
    (4, 32, 8, 128, 16, "bf16", [1200, 700, 5]),          # 16 rows
    (16, 64, 8, 128, 16, "bf16", [700, 300]),             # 128 rows
    (11, 24, 8, 128, 16, "fp16", [900, 12]),              # 33 rows
    (5, 16, 2, 64, 8, "fp16", [640, 77]),                 # 40 rows, D = 64
    (5, 12, 2, 64, 8, "fp16", [900, 300, 3]),             # 30 rows, D = 64
]


@pytest.mark.parametrize("max_ctas", [0, 3], ids=["one_cta_per_unit", "capped_grid"])
@pytest.mark.parametrize("case", VERIFY_TC, ids=[f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_{c[5]}" for c in VERIFY_TC])
def test_verify_tensor_core(case, max_ctas):
    # units of <= 32 rows: one CTA per unit runs the spread form, a capped
    # grid the one-quarter form; both raise the maximum on nearly every tile
    q_len, hq, hkv, d, bs, dt, lens = case
    kc, vc, tables, g, dtype = _pool(22, lens, hkv, d, bs, dt)
    q = torch.randn(len(lens), q_len, hq, d, generator=g, device="cuda").to(dtype)
    scale = 1 / np.sqrt(d)
    out = torch.full_like(q, float("nan"))
    ops().verify_decode_tc(q, kc, vc, torch.from_numpy(tables).cuda(),
                           torch.tensor(lens, dtype=torch.int32, device="cuda"), scale, out=out, max_ctas=max_ctas)
    _check(out, opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tables, lens, scale), f"verify tc {case}")


@pytest.mark.parametrize("bs,dt", [(16, "bf16"), (8, "fp16"), (4, "bf16")])
def test_chunked_prefill(bs, dt):
    hq, hkv, d = 16, 4, 128
    hists, chunks = [900, 0, 300], [200, 256, 37]
    lens = [h + c for h, c in zip(hists, chunks)]
    kc, vc, tables, g, dtype = _pool(23, lens, hkv, d, bs, dt)
    q = torch.randn(sum(chunks), hq, d, generator=g, device="cuda").to(dtype)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    scale = 1 / np.sqrt(d)
    out = ops().chunked_prefill(q, torch.from_numpy(q_start).cuda(), torch.tensor(lens, dtype=torch.int32,
                                device="cuda"), kc, vc, torch.from_numpy(tables).cuda(), scale, max(chunks))
    ref = opa.chunked_prefill(to_f64(q), q_start, lens, to_f64(kc), to_f64(vc), tables, scale)
    _check(out, ref, f"prefill bs {bs}")


def test_shared_prefix_decode():
    hq, hkv, d, bs, npre = 32, 8, 128, 16, 40
    rng = np.random.default_rng(24)
    lens = [int(npre * bs + s) for s in rng.integers(1, 300, size=12)]
    kc, vc, tables, g, dtype = _pool(24, lens, hkv, d, bs, "bf16", shared_blocks=npre)
    q = torch.randn(len(lens), hq, d, generator=g, device="cuda").to(dtype)
    scale = 1 / np.sqrt(d)
    t = torch.from_numpy(tables).cuda()
    out = ops().decode_shared_prefix(q, kc, vc, t[0, :npre].contiguous(), npre * bs, t,
                                     torch.tensor(lens, dtype=torch.int32, device="cuda"), scale)
    _check(out, opa.decode(to_f64(q), to_f64(kc), to_f64(vc), tables, lens, scale), "shared prefix")
