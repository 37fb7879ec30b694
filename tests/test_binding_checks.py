"""The Python binding refuses mismatched tensors before calling the library
(CPU: every check runs before a pointer is taken, so CPU tensors exercise
them).  The C calls take raw pointers and sizes; without these checks a
mismatch would be read as the wrong type, past a buffer's end, or from
another device's memory."""
import pytest
import torch

from paged_kv_cache_76_gb300 import ops
from paged_kv_cache_76_gb300 import vattention as va


def _kv(nb=4, bs=16, hkv=2, d=128, dt=torch.bfloat16):
    return torch.zeros(nb, bs, hkv, d, dtype=dt), torch.zeros(nb, bs, hkv, d, dtype=dt)


def _i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def test_cache_writes_refuse_mismatches():
    kc, vc = _kv()
    k = torch.zeros(3, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):                          # k/v dtype is not the cache's
        ops.reshape_and_cache(k.half(), k.half(), _i32(3), kc, vc)
    with pytest.raises(ValueError):                          # one slot short
        ops.reshape_and_cache(k, k, _i32(2), kc, vc)
    with pytest.raises(ValueError):                          # v_cache smaller than k_cache
        ops.reshape_and_cache(k, k, _i32(3), kc, vc[:2])
    with pytest.raises(ValueError):                          # pairs not [n, 2]
        ops.copy_blocks(kc, vc, _i32(4))
    with pytest.raises(ValueError):                          # caches of different dtypes
        ops.copy_blocks(kc, vc.half(), _i32(1, 2))


@pytest.mark.parametrize("form", ["decode", "verify", "verify_tc", "shared_prefix"])
def test_attention_calls_refuse_mismatches(form):
    kc, vc = _kv()
    B = 3
    if form in ("verify", "verify_tc"):
        q = torch.zeros(B, 4, 8, 128, dtype=torch.bfloat16)
    else:
        q = torch.zeros(B, 8, 128, dtype=torch.bfloat16)
    tables, lens = _i32(B, 2), _i32(B)

    def call(q=q, kc=kc, vc=vc, tables=tables, lens=lens, out=None):
        if form == "decode":
            return ops.decode(q, kc, vc, tables, lens, 0.1, out=out)
        if form == "verify":
            return ops.verify_decode(q, kc, vc, tables, lens, 0.1, out=out)
        if form == "verify_tc":
            return ops.verify_decode_tc(q, kc, vc, tables, lens, 0.1, out=out)
        return ops.decode_shared_prefix(q, kc, vc, _i32(1), 16, tables, lens, 0.1, out=out)

    with pytest.raises(TypeError):                           # fp16 query, bf16 cache
        call(q=q.half())
    with pytest.raises(TypeError):                           # out of another dtype
        call(out=torch.zeros_like(q, dtype=torch.float32))
    with pytest.raises(ValueError):                          # out of another shape
        call(out=torch.zeros_like(q)[:-1])
    with pytest.raises(ValueError):                          # K and V caches differ
        call(vc=vc[:, :8].contiguous())
    with pytest.raises(ValueError):                          # a table row short
        call(tables=_i32(B - 1, 2))
    with pytest.raises(ValueError):                          # tables not 2-D
        call(tables=_i32(B))
    with pytest.raises(ValueError):                          # a length short
        call(lens=_i32(B - 1))
    with pytest.raises(ValueError):                          # head_dim of q is not the cache's
        call(q=q[..., :64].contiguous())


def test_chunked_prefill_and_merge_refuse_mismatches():
    kc, vc = _kv()
    q = torch.zeros(10, 8, 128, dtype=torch.bfloat16)
    lens, q_start, tables = _i32(2), _i32(3), _i32(2, 4)
    with pytest.raises(ValueError):                          # q_start needs num_reqs + 1 entries
        ops.chunked_prefill(q, _i32(2), lens, kc, vc, tables, 0.1, 5)
    with pytest.raises(ValueError):                          # one table row per request
        ops.chunked_prefill(q, q_start, lens, kc, vc, _i32(3, 4), 0.1, 5)
    with pytest.raises(TypeError):
        ops.chunked_prefill(q.half(), q_start, lens, kc, vc, tables, 0.1, 5)
    qd = torch.zeros(3, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):                          # out of another shape
        ops.lse_merge(None, _i32(3), qd, _i32(3, 2), 16, torch.zeros(2, 8, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):                          # a length short
        ops.lse_merge(None, _i32(2), qd, _i32(3, 2), 16, torch.zeros_like(qd))


def test_contiguous_layout_calls_refuse_mismatches():
    kc = torch.zeros(4, 64, 2, 128, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    q = torch.zeros(3, 8, 128, dtype=torch.bfloat16)
    slots, lens = _i32(3), _i32(3)
    with pytest.raises(ValueError):                          # head_dim of q is not the cache's
        va.decode_contiguous(q[..., :64].contiguous(), kc, vc, slots, lens, 0.1)
    with pytest.raises(ValueError):                          # fp16 query, bf16 cache
        va.decode_contiguous(q.half(), kc, vc, slots, lens, 0.1)
    with pytest.raises(ValueError):                          # a slot id short
        va.decode_contiguous(q, kc, vc, _i32(2), lens, 0.1)
    with pytest.raises(ValueError):                          # per-slot mapped counts: one per slot
        va.decode_contiguous(q, kc, vc, slots, lens, 0.1, slot_tokens=_i32(3))
    k = torch.zeros(5, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):                          # rows not [kv_heads, head_dim] of the cache
        va.reshape_and_cache_slots(torch.zeros(5, 2, 64, dtype=torch.bfloat16),
                                   torch.zeros(5, 2, 64, dtype=torch.bfloat16), _i32(5), _i32(5), kc, vc)
    with pytest.raises(ValueError):                          # a position short
        va.reshape_and_cache_slots(k, k, _i32(5), _i32(4), kc, vc)
