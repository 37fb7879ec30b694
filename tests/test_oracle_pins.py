"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test checks the oracle against one of: a value the pages print (a
fixture under ``tests/golden/``), a library routine on a special case
(``torch.nn.functional.scaled_dot_product_attention`` in float64 on CPU,
with its own GQA grouping), a closed form, or an invariant the method must
keep (physical-permutation invariance, shared == unshared, stale data
invisible).  Together they are chosen so that a dropped term, a wrong index
or group mapping, a transposed operand or a wrong mask fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import paged_attention as pa
from oracle import sizing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sdpa(q, K, V, scale, causal=False):
    """Library attention: q [Hq, Lq, D], K/V [Hkv, L, D] float64, GQA by torch."""
    return F.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        scale=scale, is_causal=causal, enable_gqa=True)[0].numpy()


def _scatter_blocks(contig, table, num_blocks, block_size, fill=0.0):
    """Place a contiguous [L, Hkv, D] context into a pool block by block (test-side).

    Uses whole-block slices, not per-token translation, so it is a different
    route from the oracle's gather.
    """
    L, Hkv, D = contig.shape
    pool = np.full((num_blocks, block_size, Hkv, D), fill, dtype=np.float64)
    for j, b in enumerate(table):
        seg = contig[j * block_size:(j + 1) * block_size]
        pool[b, :seg.shape[0]] = seg
    return pool


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- worked example
def test_worked_example_slots_match_the_printed_table():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    p = g["printed"]
    bs = p["block_size"]
    table = p["physical_blocks"]
    # every printed logical block -> physical block, and its fill
    for lb, (lo, hi) in enumerate(p["logical_blocks"]):
        for t in range(lo, hi + 1):
            pbn, off = pa.token_location(table, t, bs)
            assert pbn == table[lb]
            assert off == t - lb * bs
        assert hi - lo + 1 == p["fill"][lb][0]
    slots = pa.slots_for(table + [99], range(12), bs)
    assert slots.tolist() == g["derived_by_hand"]["slots_tokens_0_to_11"]
    # token 12 is the first that lands in logical block 3
    assert 12 // bs == p["new_block_is_logical_block"]
    assert pa.token_location([7, 2, 5, 11], 12, bs) == (11, 0)


def test_reshape_and_cache_worked_example_roundtrip():
    rng = np.random.default_rng(3)
    bs, nb, Hkv, D = 4, 16, 1, 8
    k = _rand(rng, 9, Hkv, D)
    v = _rand(rng, 9, Hkv, D)
    slots = pa.slots_for([7, 2, 5], range(9), bs)
    kc, vc = pa.reshape_and_cache(k, v, slots, np.zeros((nb, bs, Hkv, D)), np.zeros((nb, bs, Hkv, D)))
    # test-side expectation by block slices: block 7 holds tokens 0-3, block 2 tokens 4-7, block 5 token 8
    assert np.array_equal(kc[7], k[0:4]) and np.array_equal(kc[2], k[4:8])
    assert np.array_equal(kc[5, 0], k[8]) and np.all(kc[5, 1:] == 0)
    assert np.array_equal(vc[2], v[4:8])
    untouched = [b for b in range(nb) if b not in (7, 2, 5)]
    assert np.all(kc[untouched] == 0)


def test_reshape_and_cache_skips_negative_slots_and_rejects_overflow():
    k = np.arange(2 * 1 * 4, dtype=np.float64).reshape(2, 1, 4)
    kc0 = np.full((2, 2, 1, 4), -7.0)
    kc, _ = pa.reshape_and_cache(k, k, [-1, 3], kc0, kc0)
    assert np.array_equal(kc[1, 1], k[1]) and np.all(kc.reshape(4, 4)[:3] == -7.0)
    with pytest.raises(IndexError):
        pa.reshape_and_cache(k, k, [0, 4], kc0, kc0)


def test_reshape_and_cache_is_bit_exact_on_raw_halves():
    raw = np.array([[[0x7E00, 0x8001, 0x3C00, 0xFBFF]]], dtype=np.uint16)  # NaN, -denorm, 1, -max
    kc, _ = pa.reshape_and_cache(raw, raw, [5], np.zeros((2, 4, 1, 4), np.uint16), np.zeros((2, 4, 1, 4), np.uint16))
    assert kc[1, 1].tobytes() == raw[0].tobytes()


def test_copy_blocks_copies_whole_blocks():
    rng = np.random.default_rng(0)
    kc = _rand(rng, 6, 4, 2, 8)
    vc = _rand(rng, 6, 4, 2, 8)
    k2, v2 = pa.copy_blocks(kc, vc, [(1, 4), (2, 5)])
    assert np.array_equal(k2[4], kc[1]) and np.array_equal(v2[5], vc[2])
    assert np.array_equal(k2[:4], kc[:4])
    with pytest.raises(ValueError):
        pa.copy_blocks(kc, vc, [(1, 4), (4, 5)])


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("Hq,Hkv,D,bs,L", [(2, 1, 64, 4, 9), (8, 2, 32, 16, 37), (12, 4, 16, 8, 64), (7, 7, 16, 4, 1)])
def test_decode_matches_library_attention_through_scattered_tables(Hq, Hkv, D, bs, L):
    rng = np.random.default_rng(Hq * 100 + L)
    nblk = -(-L // bs)
    nb = 3 * nblk + 5
    table = rng.permutation(nb)[:nblk].tolist()
    K = _rand(rng, L, Hkv, D)
    V = _rand(rng, L, Hkv, D)
    q = _rand(rng, Hq, D)
    scale = 1.0 / math.sqrt(D) * 1.3
    kc = _scatter_blocks(K, table, nb, bs, fill=np.nan)
    vc = _scatter_blocks(V, table, nb, bs, fill=np.nan)
    got = pa.decode(q[None], kc, vc, np.array([table]), [L], scale)[0]
    ref = _sdpa(q[:, None, :], K.transpose(1, 0, 2), V.transpose(1, 0, 2), scale)[:, 0, :]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_gqa_grouping_is_contiguous_not_interleaved():
    """With distinct KV heads, head h must use kv head h // group (library GQA)."""
    rng = np.random.default_rng(5)
    Hq, Hkv, D, bs, L = 8, 2, 16, 4, 12
    K = _rand(rng, L, Hkv, D) * 3
    V = _rand(rng, L, Hkv, D)
    V[:, 1] += 10.0  # make the two kv heads' outputs far apart
    q = _rand(rng, Hq, D)
    table = list(range(3))
    got = pa.decode(q[None], _scatter_blocks(K, table, 3, bs), _scatter_blocks(V, table, 3, bs),
                    np.array([table]), [L], 0.25)[0]
    assert np.all(got[:4].mean(axis=1) < 5) and np.all(got[4:].mean(axis=1) > 5)


def test_identity_table_equals_contiguous_attention():
    rng = np.random.default_rng(11)
    Hq, Hkv, D, bs, L = 4, 2, 16, 16, 80
    K = _rand(rng, L, Hkv, D)
    V = _rand(rng, L, Hkv, D)
    q = _rand(rng, Hq, D)
    kc = K.reshape(L // bs, bs, Hkv, D)
    vc = V.reshape(L // bs, bs, Hkv, D)
    got = pa.decode(q[None], kc, vc, np.arange(L // bs)[None], [L], 0.3)[0]
    ref = _sdpa(q[:, None], K.transpose(1, 0, 2), V.transpose(1, 0, 2), 0.3)[:, 0]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_output_invariant_under_physical_block_relabelling():
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D, bs, nb = 3, 4, 2, 16, 4, 20
    lens = [9, 13, 4]
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    perm = rng.permutation(nb)
    tables = np.array([perm[0:4], perm[4:8], perm[8:12]])
    q = _rand(rng, B, Hq, D)
    a = pa.decode(q, kc, vc, tables, lens, 0.25)
    pi = rng.permutation(nb)           # relabel: block b -> pi[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    b = pa.decode(q, kc2, vc2, pi[tables], lens, 0.25)
    assert np.array_equal(a, b)


def test_stale_data_past_the_context_is_invisible():
    """Freed / unused slots keep old data; the valid length hides it."""
    rng = np.random.default_rng(13)
    Hq, Hkv, D, bs, L, nb = 4, 1, 16, 16, 21, 4
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    table = np.array([[3, 1]])
    q = _rand(rng, 1, Hq, D)
    a = pa.decode(q, kc, vc, table, [L], 0.25)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[1, L - bs:] = np.nan
    vc2[1, L - bs:] = 1e30
    kc2[[0, 2]] = np.nan
    b = pa.decode(q, kc2, vc2, table, [L], 0.25)
    assert np.array_equal(a, b)


def test_zero_context_gives_zero_output():
    out = pa.decode(np.ones((2, 2, 4)), np.ones((2, 4, 1, 4)), np.ones((2, 4, 1, 4)),
                    np.zeros((2, 1), int), [0, 3], 1.0)
    assert np.all(out[0] == 0) and np.allclose(out[1], 1.0)


def test_prefix_shared_blocks_equal_unshared_copies():
    rng = np.random.default_rng(14)
    Hq, Hkv, D, bs = 4, 2, 16, 4
    nb = 24
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    # requests 0 and 1 share blocks 3,4 (8-token prefix) then own 10 / 11
    shared = np.array([[3, 4, 10], [3, 4, 11]])
    # unshared: request 1's prefix copied into blocks 20, 21
    kc2, vc2 = pa.copy_blocks(kc, vc, [(3, 20), (4, 21)])
    unshared = np.array([[3, 4, 10], [20, 21, 11]])
    q = _rand(rng, 2, Hq, D)
    a = pa.decode(q, kc, vc, shared, [11, 10], 0.25)
    b = pa.decode(q, kc2, vc2, unshared, [11, 10], 0.25)
    assert np.array_equal(a, b)


def test_copy_on_write_leaves_other_sharers_unchanged():
    """§6: a writer copies the shared partial block, writes the copy; others unaffected."""
    rng = np.random.default_rng(15)
    Hq, Hkv, D, bs, nb = 4, 1, 16, 4, 12
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    q = _rand(rng, 2, Hq, D)
    tables = np.array([[1, 2], [1, 2]])      # both share a 6-token context; block 2 half full
    before = pa.decode(q, kc, vc, tables, [6, 6], 0.25)
    kc2, vc2 = pa.copy_blocks(kc, vc, [(2, 7)])
    newk = _rand(rng, 1, Hkv, D)
    kc2, vc2 = pa.reshape_and_cache(newk, newk, [7 * bs + 2], kc2, vc2)  # writer appends token 6
    after = pa.decode(q, kc2, vc2, np.array([[1, 2], [1, 7]]), [6, 7], 0.25)
    assert np.array_equal(after[0], before[0])
    # the writer sees its private copy plus the new token == unshared construction
    K = np.concatenate([kc[1], kc[2, :2], newk])
    V = np.concatenate([vc[1], vc[2, :2], newk])
    ref = _sdpa(q[1][:, None], K.transpose(1, 0, 2), V.transpose(1, 0, 2), 0.25)[:, 0]
    np.testing.assert_allclose(after[1], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- split + merge
@pytest.mark.parametrize("S", [4, 8, 12, 64])
def test_split_merge_equals_direct(S):
    rng = np.random.default_rng(16)
    B, Hq, Hkv, D, bs, nb = 3, 8, 2, 16, 4, 40
    lens = [37, 5, 64]
    kc = _rand(rng, nb, bs, Hkv, D) * 2
    vc = _rand(rng, nb, bs, Hkv, D)
    perm = rng.permutation(nb)
    tables = np.array([perm[0:16], perm[16:32], perm[24:40]])
    q = _rand(rng, B, Hq, D)
    a = pa.decode(q, kc, vc, tables, lens, 0.5)
    b = pa.decode_split(q, kc, vc, tables, lens, 0.5, S)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)


def test_single_partition_partials_are_plain_softmax_terms():
    rng = np.random.default_rng(17)
    Hq, D, L = 2, 8, 9
    kc = _rand(rng, 3, 4, 1, D)
    vc = _rand(rng, 3, 4, 1, D)
    q = _rand(rng, 1, Hq, D)
    (o, m, l), = pa.decode_split_partials(q, kc, vc, np.array([[0, 1, 2]]), [L], 1.0, 512)
    K = kc.reshape(12, D)[:L]
    V = vc.reshape(12, D)[:L]
    s = K @ q[0].T                          # [L, Hq]
    np.testing.assert_allclose(m[0], s.max(axis=0), atol=1e-14)
    np.testing.assert_allclose(l[0], np.exp(s - s.max(axis=0)).sum(axis=0), rtol=1e-13)
    # merge of a single partition is o / l
    np.testing.assert_allclose(pa.lse_merge(o, m, l), o[0] / l[0][:, None], rtol=1e-13)


def test_lse_merge_is_invariant_to_shifting_a_partition():
    """Shifting m_c by d while scaling o_c, l_c by exp(-d) describes the same partition."""
    rng = np.random.default_rng(18)
    o = _rand(rng, 3, 5)
    m = _rand(rng, 3)
    l = np.abs(_rand(rng, 3)) + 0.5
    a = pa.lse_merge(o, m, l)
    d = np.array([3.0, -40.0, 0.7])
    b = pa.lse_merge(o * np.exp(-d)[:, None], m + d, l * np.exp(-d))
    np.testing.assert_allclose(a, b, rtol=1e-12)


# ---------------------------------------------------------------- chunked prefill
def _prefill_case(rng, Hq, Hkv, D, bs, L, nb):
    nblk = -(-L // bs)
    table = rng.permutation(nb)[:nblk]
    K = _rand(rng, L, Hkv, D)
    V = _rand(rng, L, Hkv, D)
    return table, K, V, _scatter_blocks(K, table, nb, bs), _scatter_blocks(V, table, nb, bs)


def test_prefill_without_history_is_causal_attention():
    rng = np.random.default_rng(19)
    Hq, Hkv, D, bs, L = 6, 2, 16, 4, 13
    table, K, V, kc, vc = _prefill_case(rng, Hq, Hkv, D, bs, L, 10)
    q = _rand(rng, L, Hq, D)
    got = pa.chunked_prefill(q, [0, L], [L], kc, vc, np.array([table]), 0.3)
    ref = _sdpa(q.transpose(1, 0, 2), K.transpose(1, 0, 2), V.transpose(1, 0, 2), 0.3, causal=True)
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_prefill_chunk_over_history_equals_rows_of_full_causal_attention():
    rng = np.random.default_rng(20)
    Hq, Hkv, D, bs = 4, 1, 16, 8
    L, chunk = 29, 7
    table, K, V, kc, vc = _prefill_case(rng, Hq, Hkv, D, bs, L, 12)
    qfull = _rand(rng, L, Hq, D)
    full = _sdpa(qfull.transpose(1, 0, 2), K.transpose(1, 0, 2), V.transpose(1, 0, 2), 0.4, causal=True)
    got = pa.chunked_prefill(qfull[L - chunk:], [0, chunk], [L], kc, vc, np.array([table]), 0.4)
    np.testing.assert_allclose(got, full.transpose(1, 0, 2)[L - chunk:], rtol=1e-12, atol=1e-12)


def test_prefill_chunk_of_one_is_decode_and_requests_are_independent():
    rng = np.random.default_rng(21)
    Hq, Hkv, D, bs, nb = 4, 2, 16, 4, 30
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    perm = rng.permutation(nb)
    tables = np.array([perm[:6], perm[6:12]])
    q = _rand(rng, 1 + 3, Hq, D)
    got = pa.chunked_prefill(q, [0, 1, 4], [17, 22], kc, vc, tables, 0.3)
    dec = pa.decode(q[:1], kc, vc, tables[:1], [17], 0.3)
    np.testing.assert_allclose(got[0], dec[0], rtol=1e-13, atol=1e-13)
    # request 1's last query sees its whole context: decode of the same query
    dec1 = pa.decode(q[3:4], kc, vc, tables[1:2], [22], 0.3)
    np.testing.assert_allclose(got[3], dec1[0], rtol=1e-13, atol=1e-13)
    dec1b = pa.decode(q[1:2], kc, vc, tables[1:2], [20], 0.3)
    np.testing.assert_allclose(got[1], dec1b[0], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- speculative verify
@pytest.mark.parametrize("Q,Hq,Hkv,L", [(4, 8, 2, 37), (1, 4, 4, 9), (8, 6, 3, 8), (3, 4, 1, 100)])
def test_verify_decode_is_the_last_rows_of_library_causal_attention(Q, Hq, Hkv, L):
    """The k+1 queries of a request are the last k+1 rows of causal attention
    over the whole context (torch's SDPA on contiguous K/V, GQA by torch)."""
    rng = np.random.default_rng(40 + Q)
    D, bs = 16, 4
    table, K, V, kc, vc = _prefill_case(rng, Hq, Hkv, D, bs, L, 40)
    qfull = _rand(rng, L, Hq, D)
    full = _sdpa(qfull.transpose(1, 0, 2), K.transpose(1, 0, 2), V.transpose(1, 0, 2), 0.35, causal=True)
    q = qfull[L - Q:][None]                                   # [1, Q, Hq, D]
    got = pa.verify_decode(q, kc, vc, np.array([table]), [L], 0.35)
    np.testing.assert_allclose(got[0], full.transpose(1, 0, 2)[L - Q:], rtol=1e-12, atol=1e-12)


def test_verify_decode_batches_requests_and_its_last_query_is_decode():
    rng = np.random.default_rng(44)
    Hq, Hkv, D, bs, nb, Q = 4, 2, 16, 4, 40, 3
    kc = _rand(rng, nb, bs, Hkv, D)
    vc = _rand(rng, nb, bs, Hkv, D)
    perm = rng.permutation(nb)
    tables = np.array([perm[:8], perm[8:16]])
    lens = [29, 13]
    q = _rand(rng, 2, Q, Hq, D)
    got = pa.verify_decode(q, kc, vc, tables, lens, 0.3)
    for r in range(2):
        for i in range(Q):
            dec = pa.decode(q[r, i][None], kc, vc, tables[r:r + 1], [lens[r] - (Q - 1 - i)], 0.3)
            np.testing.assert_allclose(got[r, i], dec[0], rtol=1e-13, atol=1e-13)


def test_verify_decode_queries_before_the_first_key_give_zero_rows():
    rng = np.random.default_rng(45)
    Hq, Hkv, D, bs, Q = 2, 1, 8, 4, 5
    kc = _rand(rng, 6, bs, Hkv, D)
    vc = _rand(rng, 6, bs, Hkv, D)
    q = _rand(rng, 1, Q, Hq, D)
    got = pa.verify_decode(q, kc, vc, np.array([[3, 1]]), [3], 0.5)  # queries 0, 1 see nothing
    assert not got[0, :2].any()
    # query 2 sees exactly one key: its output is that key's value row, for every head
    np.testing.assert_allclose(got[0, 2], np.repeat(vc[3, 0, 0][None], Hq, 0), atol=1e-15)


# ---------------------------------------------------------------- sizing
def test_kv_size_closed_form_matches_the_printed_numbers():
    g = json.load(open(os.path.join(GOLDEN, "kv_sizing.json")))
    s = g["per_layer_k_or_v_slot"]
    S = sizing.kv_slot_bytes(s["length"], s["kv_heads"], s["head_dim"], s["elem_bytes"])
    assert S == s["exact_bytes"]
    assert abs(S / 1e6 - 200) < 5                            # "~200 MB"
    v = g["virtual_reservation"]
    assert abs(v["batch"] * S / 1e9 - v["printed_per_layer_tensor_gb"]) < 3   # B*S ~ 100 GB
    total = 2 * v["layers"] * v["batch"] * S                  # K and V, all layers
    assert abs(total / 1e12 - v["printed_total_tb"]) < 0.5
    # M_KV = 2 N L H D P for one request of full length == K+V over layers
    assert sizing.kv_cache_bytes(60, 200000, 4, 128, 2) == 2 * 60 * S
    t = g["tail_commit"]
    assert 2 * t["layers"] * t["page_mb"] == t["printed_mb"]


def _touched_bytes(tables, lens, Hq, Hkv, D, bs, q_len, nb, unique):
    """Brute force: mark every array element one decode step reads or writes.

    Real arrays of the step's dtypes (fp16 cache, q and out; int32 tables and
    lengths) get one boolean mask each; every (request, logical token) marks
    its K and V rows through the Block Table, and each request marks its
    query and output rows, the table entries that cover its tokens and its
    length.  Bytes = marked elements x itemsize, summed over the arrays.
    With ``unique`` the K/V masks are shared by the batch (a row read twice
    counts once); otherwise every request gets fresh K/V masks.
    """
    B = len(lens)
    arrays = {
        "k": np.zeros((nb, bs, Hkv, D), np.float16), "v": np.zeros((nb, bs, Hkv, D), np.float16),
        "q": np.zeros((B, q_len, Hq, D), np.float16), "o": np.zeros((B, q_len, Hq, D), np.float16),
        "table": np.asarray(tables, np.int32), "lens": np.asarray(lens, np.int32),
    }
    total = 0

    def fresh(names):
        return {n: np.zeros(arrays[n].shape, bool) for n in names}

    masks = fresh(arrays)
    for r in range(B):
        if not unique and r:
            for n, m in fresh(["k", "v"]).items():
                total += int(masks[n].sum()) * arrays[n].itemsize
                masks[n] = m
        for t in range(int(lens[r])):
            blk = int(arrays["table"][r][t // bs])
            masks["k"][blk, t % bs] = True
            masks["v"][blk, t % bs] = True
            masks["table"][r, t // bs] = True
        masks["q"][r] = True
        masks["o"][r] = True
        masks["lens"][r] = True
    for n, m in masks.items():
        total += int(m.sum()) * arrays[n].itemsize
    return total


@pytest.mark.parametrize("q_len", [1, 4])
def test_decode_step_bytes_equals_a_count_of_touched_elements(q_len):
    rng = np.random.default_rng(11)
    Hq, Hkv, D, bs, nb = 6, 2, 8, 4, 40
    lens = [1, 4, 5, 13, 0, 9]
    perm = rng.permutation(nb)
    tables, k = [], 0
    for L in lens:  # private blocks for every request: no row is shared
        n = -(-L // bs)
        tables.append(list(perm[k:k + n]) + [-1] * (4 - n))
        k += n
    want = _touched_bytes(tables, lens, Hq, Hkv, D, bs, q_len, nb, unique=False)
    assert sizing.decode_step_bytes(lens, Hq, Hkv, D, bs, 2, q_len) == want
    # nothing shared: every row is unique, so the two counts agree
    assert sizing.unique_kv_bytes(tables, lens, Hq, Hkv, D, bs, 2, q_len) == want
    assert _touched_bytes(tables, lens, Hq, Hkv, D, bs, q_len, nb, unique=True) == want


def test_unique_kv_bytes_counts_a_shared_prefix_once():
    """"2.1 PagedAttention" §6: Block Tables of several requests point at one
    prefix.  Three requests share two full blocks and a third, partial one
    (read to different depths); each has a private tail."""
    Hq, Hkv, D, bs, nb = 4, 1, 8, 4, 16
    shared = [3, 7, 9]
    tables = [shared + [0, -1], shared + [5, 6], shared + [-1, -1]]
    lens = [13, 19, 10]      # tokens 0-7 (blocks 3, 7) by all; block 9 to depth 4, 4, 2
    brute = _touched_bytes(tables, lens, Hq, Hkv, D, bs, 1, nb, unique=True)
    assert sizing.unique_kv_bytes(tables, lens, Hq, Hkv, D, bs) == brute
    # by hand: distinct rows = 8 (blocks 3, 7) + 4 (block 9) + 1 (block 0) + 4 + 3 (blocks 5, 6) = 20
    row = 2 * Hkv * D * 2
    per_req = sum(2 * Hq * D * 2 + 4 * (-(-L // bs)) + 4 for L in lens)
    assert brute == 20 * row + per_req
    # the logical count reads the shared rows once per request
    assert sizing.decode_step_bytes(lens, Hq, Hkv, D, bs) == sum(lens) * row + per_req


def test_unique_kv_bytes_of_a_2048_token_shared_prefix():
    """The prefix-shared decode shape: a 2048-token prefix is 128 blocks of 16
    tokens held by every request (refcount = batch), then private suffixes.
    Closed form: (2048 + sum of suffixes) K+V rows, plus the per-request terms."""
    Hq, Hkv, D, bs = 4, 2, 8, 16
    prefix_blocks = list(range(100, 228))
    assert len(prefix_blocks) * bs == 2048
    suffix = [16, 17, 40, 512, 1]
    tables, nxt = [], 1000
    for s in suffix:
        n = -(-s // bs)
        tables.append(prefix_blocks + list(range(nxt, nxt + n)))
        nxt += n
    lens = [2048 + s for s in suffix]
    row = 2 * Hkv * D * 2
    per_req = sum(2 * Hq * D * 2 + 4 * (-(-L // bs)) + 4 for L in lens)
    assert sizing.unique_kv_bytes(tables, lens, Hq, Hkv, D, bs) == (2048 + sum(suffix)) * row + per_req
    assert sizing.decode_step_bytes(lens, Hq, Hkv, D, bs) == (5 * 2048 + sum(suffix)) * row + per_req
