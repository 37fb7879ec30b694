"""The workload scripts replay cleanly on the oracle allocator and have the stated shape."""
import numpy as np
import pytest

import workloads as W
from oracle.block_pool import SequenceManager


def _replay(wl):
    m = SequenceManager(wl.num_blocks, wl.block_size, wl.free_order)
    m.run(wl.setup_ops)
    slots, pairs = m.run(wl.step_ops)
    return m, slots, pairs


def test_tiny_workload_reproduces_the_worked_example_table():
    wl = W.tiny_paged_decode()
    m, slots, pairs = _replay(wl)
    assert m.block_table(0) == [7, 2, 5]
    assert slots[:9] == [28, 29, 30, 31, 8, 9, 10, 11, 20]
    assert len(slots) == 14 and wl.new_tokens == 14 and pairs == []


@pytest.mark.parametrize("name", ["llama8b_gqa_decode", "long_context_splitk_decode"])
def test_decode_workloads_shape(name):
    wl = W.WORKLOADS[name]()
    m, slots, pairs = _replay(wl)
    assert len(slots) == len(wl.decode_seqs) == wl.new_tokens
    for s, L in zip(wl.decode_seqs, wl.decode_lens):
        assert m.num_tokens[s] == L and len(m.block_table(s)) == -(-L // wl.block_size)
    used = sum(len(m.block_table(s)) for s in wl.decode_seqs)
    assert wl.num_blocks == int(np.ceil(1.5 * used))
    lo, hi = (512, 4096) if name.startswith("llama") else (32768, 131072)
    assert lo <= min(wl.decode_lens) and max(wl.decode_lens) <= hi


def test_spec_verify_workload_writes_k_plus_one_tokens_per_request():
    wl = W.spec_verify_decode()
    m, slots, pairs = _replay(wl)
    assert wl.q_len == 4 and len(slots) == wl.new_tokens == 4 * len(wl.decode_seqs) and pairs == []
    for s, L in zip(wl.decode_seqs, wl.decode_lens):
        assert m.num_tokens[s] == L and 512 <= L <= 4096
    vals = W.make_values(wl)
    assert vals["q_decode"].shape == (64, 4, 32, 128)


def test_prefix_shared_workload_refcounts_and_cow():
    wl = W.prefix_shared_cow_decode()
    m = SequenceManager(wl.num_blocks, wl.block_size, wl.free_order)
    m.run(wl.setup_ops)
    prefix = m.block_table(0)[:128]
    assert all(m.ref(b) == 256 for b in prefix)
    assert all(m.block_table(r)[:128] == prefix for r in range(256))
    _, pairs = m.run(wl.step_ops)
    assert len(pairs) == 26 and all(s == prefix[127] for s, _ in pairs)
    assert m.ref(prefix[127]) == 256 - 26
    assert len({d for _, d in pairs}) == 26


def test_mixed_workload_has_prefill_chunks_and_decodes():
    wl = W.mixed_prefill_decode()
    m, slots, _ = _replay(wl)
    assert len(wl.prefill) == 4 and all(c == 512 for _, c, _ in wl.prefill)
    assert wl.new_tokens == 4 * 512 + 192 == len(slots)
    for s, c, L in wl.prefill:
        assert m.num_tokens[s] == L and 512 <= L <= 8192 + 512


def test_values_are_seeded_and_shaped():
    wl = W.tiny_paged_decode()
    a = W.make_values(wl)
    b = W.make_values(wl)
    assert all(torch_equal(a[k], b[k]) for k in a)
    assert a["k_cache"].shape == (16, 4, 1, 64) and a["q_decode"].shape == (2, 2, 64)
    assert a["k_new"].shape == (14, 1, 64)
    assert float(a["q_decode"].float().abs().max()) <= 1.0


def torch_equal(x, y):
    return bool((x.view(-1).view(dtype=__import__("torch").int16) == y.view(-1).view(dtype=__import__("torch").int16)).all())
