"""Speculative verify attention on the GPU ("Khám phá vLLM … phần 2",
speculative decoding): k+1 queries per request over the paged cache, against
the float64 oracle, plus the bitwise identities the method fixes (query i is
decode over the first L-k+i tokens; q_len = 1 is decode)."""
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


def _case(seed, q_len, hq, hkv, d, bs, dt, lens, extra_blocks=3):
    rng = np.random.default_rng(seed)
    nblk = [max(-(-L // bs), 1) for L in lens]
    maxblk = max(nblk) + extra_blocks
    nb = sum(nblk) + 7
    perm = rng.permutation(nb)
    tables = np.full((len(lens), maxblk), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(nblk):
        tables[r, :n] = perm[off:off + n]
        off += n
    g = torch.Generator(device="cuda").manual_seed(seed)
    dtype = torch.bfloat16 if dt == "bf16" else torch.float16
    kc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(dtype)
    vc = torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(dtype)
    q = torch.randn(len(lens), q_len, hq, d, generator=g, device="cuda").to(dtype)
    return q, kc, vc, torch.from_numpy(tables).cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda")


VERIFY_CASES = [
    # q_len, q_heads, kv_heads, head_dim, block_size, dtype, lens, split_tokens
    (4, 32, 8, 128, 16, "bf16", [700, 4, 1025, 33, 16], 0),         # 16 columns
    (8, 32, 8, 128, 16, "bf16", [2000, 9, 517, 8], 256),           # 32 columns; last partitions empty for early queries
    (3, 8, 8, 64, 4, "fp16", [2, 3, 50, 1], 64),                   # contexts shorter than q_len: zero rows
    (2, 16, 2, 128, 32, "bf16", [1000, 65, 64], 128),
    (5, 12, 2, 64, 8, "fp16", [300, 77, 5], 0),                    # 30 columns
    (6, 4, 1, 128, 16, "bf16", [4096, 3000], 512),                 # 24 columns, many partitions
    (1, 28, 4, 128, 16, "bf16", [300, 1029], 256),                 # q_len 1
    # 16-token partitions: more than 32 per row (the block-per-row merge)
    (4, 32, 8, 128, 16, "bf16", [512, 2000, 515, 3], 16),
    (4, 16, 4, 64, 16, "fp16", [1500, 40, 513], 16),
    (8, 32, 8, 128, 16, "bf16", [1030, 9, 600], 16),
]


@pytest.mark.parametrize("case", VERIFY_CASES, ids=[f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}" for c in VERIFY_CASES])
def test_verify_matches_the_oracle(case):
    q_len, hq, hkv, d, bs, dt, lens, split = case
    q, kc, vc, tables, lens_t = _case(1, q_len, hq, hkv, d, bs, dt, lens)
    scale = 1 / np.sqrt(d)
    out = ops().verify_decode(q, kc, vc, tables, lens_t, scale, split_tokens=split)
    ref = opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tables.cpu().numpy(), lens, scale)
    assert_close(out, ref, f"verify {case}")
    for r, L in enumerate(lens):
        for i in range(q_len):
            if L - (q_len - 1 - i) <= 0:
                assert torch.count_nonzero(out[r, i]) == 0
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_verify_with_exactly_32_partitions(dt):
    """The widest table covers 512 tokens in 16-token partitions: 32 partitions,
    the one-warp merge at its limit (lane c = partition c)."""
    q_len, hq, hkv, d, bs = 4, 32, 8, 128, 16
    lens = [512, 509, 100, 4]
    q, kc, vc, tables, lens_t = _case(6, q_len, hq, hkv, d, bs, dt, lens, extra_blocks=0)
    assert tables.shape[1] * bs // 16 == 32
    scale = 1 / np.sqrt(d)
    out = ops().verify_decode(q, kc, vc, tables, lens_t, scale, split_tokens=16)
    ref = opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tables.cpu().numpy(), lens, scale)
    assert_close(out, ref, f"verify 32 partitions {dt}")
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("split", [0, 128])
def test_each_query_is_bitwise_decode_over_its_visible_prefix(split):
    q_len, hq, hkv, d, bs = 7, 32, 8, 128, 16
    lens = [900, 130, 129, 7, 2050]
    q, kc, vc, tables, lens_t = _case(2, q_len, hq, hkv, d, bs, "bf16", lens)
    scale = 1 / np.sqrt(d)
    out = ops().verify_decode(q, kc, vc, tables, lens_t, scale, split_tokens=split)
    # the same partitions as the verify call (its automatic choice differs from decode's)
    dsplit = ops().verify_split_tokens(tables.shape[1], bs, q_len, split)
    for i in range(q_len):
        li = torch.clamp(lens_t - (q_len - 1 - i), min=0).to(torch.int32)
        dec = ops().decode(q[:, i].contiguous(), kc, vc, tables, li, scale, split_tokens=dsplit)
        assert torch.equal(out[:, i], dec), i
    assert ops().get_device_error() == 0


def test_q_len_one_is_decode_bitwise_and_relabelling_changes_no_bit():
    hq, hkv, d, bs = 32, 8, 128, 16
    lens = [1500, 17, 600]
    q, kc, vc, tables, lens_t = _case(3, 1, hq, hkv, d, bs, "bf16", lens)
    scale = 1 / np.sqrt(d)
    out = ops().verify_decode(q, kc, vc, tables, lens_t, scale)
    assert torch.equal(out[:, 0], ops().decode(q[:, 0].contiguous(), kc, vc, tables, lens_t, scale))
    q4, kc4, vc4, t4, l4 = _case(4, 4, hq, hkv, d, bs, "bf16", lens)
    a = ops().verify_decode(q4, kc4, vc4, t4, l4, scale)
    pi = torch.randperm(kc4.shape[0], generator=torch.Generator().manual_seed(5)).cuda()
    k2, v2 = torch.empty_like(kc4), torch.empty_like(vc4)
    k2[pi] = kc4
    v2[pi] = vc4
    t2 = torch.where(t4 >= 0, pi[t4.clamp(min=0).long()].int(), t4)
    b = ops().verify_decode(q4, k2, v2, t2, l4, scale)
    assert torch.equal(a, b)
    assert ops().get_device_error() == 0


def test_verify_rejects_too_many_columns_and_bad_q_len():
    from paged_kv_cache_76_gb300 import _lib
    q, kc, vc, tables, lens_t = _case(6, 3, 48, 4, 128, 16, "bf16", [40])   # 12 heads x 3 queries = 36 columns
    with pytest.raises(_lib.PAError):
        ops().verify_decode(q, kc, vc, tables, lens_t, 0.1)
    L = _lib.lib()
    st = L.pa_verify_decode(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), tables.shape[1],
                            lens_t.data_ptr(), 1, 0, 48, 4, 128, 16, kc.shape[0], 0.1, 0, None, 0, q.data_ptr(),
                            _lib.PA_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PA_ERR_INVALID
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("q_len,split", [(1, 256), (4, 0), (8, 128)])
def test_rising_scores_move_the_reference_per_column(q_len, split):
    # K grows along each request's context, so every column's maximum keeps
    # rising past its exponent reference, at different tiles for different
    # columns: the output still matches the oracle, and each query still
    # equals decode over its visible prefix bit for bit (a column's
    # reference never depends on its neighbours).
    hq, hkv, d, bs = 32, 8, 128, 16
    lens = [1500, 37, 700]
    q, kc, vc, tables, lens_t = _case(11, q_len, hq, hkv, d, bs, "bf16", lens)
    tab = tables.cpu().numpy()
    grow = torch.ones(kc.shape[0], device="cuda")
    for r, L in enumerate(lens):
        for j in range(-(-L // bs)):
            grow[int(tab[r, j])] = 1.0 + 0.35 * j
    kc = (kc.float() * grow[:, None, None, None]).to(kc.dtype)
    scale = 1 / np.sqrt(d)
    out = ops().verify_decode(q, kc, vc, tables, lens_t, scale, split_tokens=split)
    ref = opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tab, lens, scale)
    assert_close(out, ref, f"rising scores q_len {q_len}")
    dsplit = ops().verify_split_tokens(tables.shape[1], bs, q_len, split)
    for i in range(q_len):
        li = torch.clamp(lens_t - (q_len - 1 - i), min=0).to(torch.int32)
        dec = ops().decode(q[:, i].contiguous(), kc, vc, tables, li, scale, split_tokens=dsplit)
        assert torch.equal(out[:, i], dec), i
    assert ops().get_device_error() == 0


# ---------------------------------------------------------------- tensor-core form (pa_verify_decode_tc)
TC_CASES = [c for c in VERIFY_CASES if c[4] >= 8 and (c[1] // c[2]) * c[0] <= 128] + [
    # q_len, q_heads, kv_heads, head_dim, block_size, dtype, lens, split_tokens (unused)
    (8, 32, 8, 128, 16, "bf16", [2339, 130, 17, 4096, 1], 0),      # the k = 7 workload's shape: 32 rows
    (16, 64, 8, 128, 16, "bf16", [700, 129, 300], 0),              # 128 rows: a full tile
    (4, 28, 4, 128, 8, "fp16", [1000, 33, 257, 2], 0),             # 28 rows, 8-token blocks
    (5, 16, 2, 64, 32, "bf16", [640, 77, 3], 0),                   # D = 64, 32-token blocks
    (8, 64, 8, 128, 16, "bf16", [900, 5, 64], 0),                  # 64 rows: two lane quarters, all full
    (11, 24, 8, 128, 16, "fp16", [300, 12, 1], 0),                 # 33 rows: the second quarter holds one
    (13, 40, 8, 64, 8, "bf16", [500, 20], 0),                      # 65 rows: one 128-row unit per CTA
]


@pytest.mark.parametrize("max_ctas", [0, 2], ids=["one_cta_per_unit", "capped_grid"])
@pytest.mark.parametrize("case", TC_CASES, ids=[f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}_{c[5]}" for c in TC_CASES])
def test_verify_tc_matches_the_oracle(case, max_ctas):
    # <= 32 rows: the spread form (one CTA per unit) and the one-quarter form
    # (a capped grid, several units per CTA)
    q_len, hq, hkv, d, bs, dt, lens, _ = case
    q, kc, vc, tables, lens_t = _case(7, q_len, hq, hkv, d, bs, dt, lens)
    scale = 1 / np.sqrt(d)
    out = torch.full_like(q, float("nan"))
    ops().verify_decode_tc(q, kc, vc, tables, lens_t, scale, out=out, max_ctas=max_ctas)
    ref = opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tables.cpu().numpy(), lens, scale)
    assert_close(out, ref, f"verify tc {case}")
    for r, L in enumerate(lens):
        for i in range(q_len):
            if L - (q_len - 1 - i) <= 0:
                assert torch.count_nonzero(out[r, i]) == 0
    assert ops().get_device_error() == 0


@pytest.mark.parametrize("q_len,hq", [(8, 32), (16, 32)], ids=["32rows", "64rows"])
def test_verify_tc_persistent_grid_matches_one_cta_per_unit_and_the_mma_form(q_len, hq):
    # 64 rows: both grids run the same per-unit arithmetic, so the bits are
    # equal.  32 rows: one CTA per unit spreads the rows over the four lane
    # quarters (merged partials), a capped grid keeps them in one quarter:
    # both within the tolerance of the oracle.
    hkv, d, bs = 8, 128, 16
    lens = [3000, 1, 6, 700, 129, 4096, 2048, 17, 900]
    q, kc, vc, tables, lens_t = _case(8, q_len, hq, hkv, d, bs, "bf16", lens)
    scale = 1 / np.sqrt(d)
    a = ops().verify_decode_tc(q, kc, vc, tables, lens_t, scale)
    b = ops().verify_decode_tc(q, kc, vc, tables, lens_t, scale, max_ctas=5)
    if q_len * hq // hkv > 32:
        assert torch.equal(a, b)
    else:
        # contexts of 1 to 17 tokens leave some queries a softmax over a few
        # keys, whose output is close to a V row of magnitude up to ~4: the
        # bound admits the output's own rounding to bf16 on top of 1e-2
        ref = opa.verify_decode(to_f64(q), to_f64(kc), to_f64(vc), tables.cpu().numpy(), lens, scale)
        assert_close(a, ref, "one CTA per unit", rounding=True)
        assert_close(b, ref, "capped grid", rounding=True)
    if q_len * hq // hkv <= 32:  # the warp-MMA form takes up to 32 columns
        m = ops().verify_decode(q, kc, vc, tables, lens_t, scale)
        err = (to_f64(a) - to_f64(m))
        assert np.abs(err).max() <= 2 * 1e-2 and np.abs(err).mean() <= 1e-3
    assert ops().get_device_error() == 0


def test_verify_tc_argument_checks():
    from paged_kv_cache_76_gb300 import _lib
    q, kc, vc, tables, lens_t = _case(9, 8, 32, 8, 128, 16, "bf16", [100, 200])
    with pytest.raises(_lib.PAError):                       # 17 queries x 8 group heads > 128 rows
        q2 = torch.zeros(2, 17, 64, 128, dtype=torch.bfloat16, device="cuda")
        ops().verify_decode_tc(q2, kc, vc, tables, lens_t, 0.1)
    q4, kc4, vc4, t4, l4 = _case(9, 4, 8, 8, 64, 4, "fp16", [50, 60])
    with pytest.raises(_lib.PAError):                       # 4-token blocks: no tcgen05 gather
        ops().verify_decode_tc(q4, kc4, vc4, t4, l4, 0.1)
    assert ops().get_device_error() == 0
