"""The C-ABI library loads here (no GPU needed) and exports every declared call."""
import os
import re

import pytest

from paged_kv_cache_76_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    try:
        return _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()
        return _lib.lib()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


def test_binding_prototypes_cover_the_header():
    assert set(_lib.PROTOTYPES) == set(declared_functions())


def test_host_only_calls(lib):
    assert lib.pa_version() >= 100
    assert lib.pa_status_string(-2) == b"PA_ERR_NO_FREE_BLOCKS"
    assert lib.pa_status_string(-8) == b"PA_ERR_HOST_MEMORY"
    with pytest.raises(MemoryError):                      # the binding raises it as a MemoryError
        _lib.check(_lib.PA_ERR_HOST_MEMORY, "probe")
    assert lib.pa_decode_split_tokens(256, 16, 0) == 384          # auto, contexts up to 8K
    assert lib.pa_decode_split_tokens(1024, 16, 0) == 512         # auto, longer contexts
    assert lib.pa_decode_split_tokens(256, 16, 24) == _lib.PA_ERR_INVALID      # not a multiple of 16
    assert lib.pa_decode_split_tokens(256, 32, 48) == _lib.PA_ERR_INVALID      # not a multiple of bs=32
    assert lib.pa_decode_split_tokens(256, 4, 2048) == _lib.PA_ERR_INVALID     # > 256 * bs
    assert lib.pa_verify_split_tokens(256, 16, 4, 0) == 768           # verify auto, contexts up to 8K
    assert lib.pa_verify_split_tokens(256, 32, 8, 0) == 768
    assert lib.pa_verify_split_tokens(256, 16, 1, 0) == 384           # q_len 1 is decode
    assert lib.pa_verify_split_tokens(1024, 16, 4, 0) == 512          # longer contexts: decode's choice
    assert lib.pa_verify_split_tokens(256, 16, 4, 128) == 128         # explicit
    assert lib.pa_verify_split_tokens(256, 16, 0, 0) == _lib.PA_ERR_INVALID
    assert lib.pa_verify_split_tokens(256, 16, 4, 24) == _lib.PA_ERR_INVALID
    assert lib.pa_selftest_wait_timeout(0, None) == _lib.PA_ERR_INVALID        # limits checked on the host
    assert lib.pa_selftest_wait_timeout(2001, None) == _lib.PA_ERR_INVALID
    # shared-prefix suffixes: a quarter of the suffix bound, >= 128, <= the decode default
    assert lib.pa_decode_shared_prefix_split_tokens(160, 16, 2048, 0) == 128    # suffix bound 512
    assert lib.pa_decode_shared_prefix_split_tokens(256, 16, 1024, 0) == 384    # bound 3072 -> 768, capped
    assert lib.pa_decode_shared_prefix_split_tokens(114, 16, 1024, 0) == 208    # bound 800 -> 200 -> 208
    assert lib.pa_decode_shared_prefix_split_tokens(160, 16, 2048, 64) == 64    # explicit
    assert lib.pa_decode_shared_prefix_split_tokens(160, 16, 2050, 0) == _lib.PA_ERR_INVALID
    # one partition needs no scratch; several need o + m + l per (seq, head, partition)
    assert lib.pa_decode_workspace_size(64, 32, 128, 24, 16, 0) == 0
    ws = lib.pa_decode_workspace_size(8, 64, 128, 8192, 16, 512)
    rows = 8 * 64 * 256
    assert ws >= rows * (128 + 2) * 4 and ws < rows * (128 + 2) * 4 + 1024


def test_device_calls_reject_bad_arguments_before_launching(lib):
    # invalid shapes are caught on the host (no GPU touched): bad head_dim, bad block size, bad dtype
    assert lib.pa_reshape_and_cache(None, None, None, 1, None, None, 4, 16, 1, 96, 1, None) == _lib.PA_ERR_INVALID
    assert lib.pa_copy_blocks(None, None, None, 1, 4, 12, 1, 64, 1, None) == _lib.PA_ERR_INVALID
    assert lib.pa_copy_blocks(None, None, None, 1, 4, 16, 1, 64, 7, None) == _lib.PA_ERR_DTYPE
    # zero-size work is a no-op that needs no pointers
    assert lib.pa_reshape_and_cache(None, None, None, 0, None, None, 4, 16, 1, 64, 1, None) == _lib.PA_OK
    assert lib.pa_decode(None, None, None, None, 4, None, 0, 8, 2, 128, 16, 4, 0.1, 0, None, 0, None, 1,
                         None) == _lib.PA_OK
    # q_heads not a multiple of kv_heads, or group > 16
    assert lib.pa_decode(1, 1, 1, 1, 4, 1, 1, 6, 4, 128, 16, 4, 0.1, 0, None, 0, 1, 1, None) == _lib.PA_ERR_INVALID
    assert lib.pa_decode(1, 1, 1, 1, 4, 1, 1, 34, 2, 128, 16, 4, 0.1, 0, None, 0, 1, 1, None) == _lib.PA_ERR_INVALID
    # a split context without a workspace
    assert lib.pa_decode(16, 16, 16, 16, 64, 16, 1, 8, 2, 128, 16, 4, 0.1, 512, None, 0, 16, 1,
                         None) == _lib.PA_ERR_WORKSPACE
    # misaligned device pointer
    assert lib.pa_decode(17, 16, 16, 16, 4, 16, 1, 8, 2, 128, 16, 4, 0.1, 0, None, 0, 16, 1,
                         None) == _lib.PA_ERR_INVALID


def test_newer_calls_reject_bad_arguments_before_touching_the_gpu(lib):
    inv = _lib.PA_ERR_INVALID
    # swap: bad head_dim / dtype, negative pair count; zero pairs is a no-op
    assert lib.pa_swap_blocks(None, None, None, None, None, 1, 4, 4, 16, 1, 96, 1, None) == inv
    assert lib.pa_swap_blocks(None, None, None, None, None, 1, 4, 4, 16, 1, 64, 9, None) == _lib.PA_ERR_DTYPE
    assert lib.pa_swap_blocks(None, None, None, None, None, -1, 4, 4, 16, 1, 64, 1, None) == inv
    assert lib.pa_swap_blocks(None, None, None, None, None, 0, 4, 4, 16, 1, 64, 1, None) == _lib.PA_OK
    # verify: q_len < 1, or more than 32 (query, group head) columns per KV head
    args = (16, 16, 16, 16, 8, 16, 1)
    assert lib.pa_verify_decode(*args, 0, 8, 2, 128, 16, 4, 0.1, 0, None, 0, 16, 1, None) == inv
    assert lib.pa_verify_decode(*args, 9, 8, 2, 128, 16, 4, 0.1, 0, None, 0, 16, 1, None) == inv   # 4 x 9 = 36
    assert lib.pa_verify_workspace_size(4, 0, 8, 128, 8, 16, 0) == 0
    n1 = lib.pa_verify_workspace_size(4, 1, 8, 128, 64, 16, 128)
    assert n1 > 0 and lib.pa_verify_workspace_size(4, 3, 8, 128, 64, 16, 128) >= 3 * n1 - 2048
    # contiguous decode / slot writes: max_len not a multiple of 16, no slots
    assert lib.pa_decode_contiguous(16, 16, 16, 4, 100, None, None, 16, 1, 8, 2, 128, 0.1, 0, None, 0, 16, 1,
                                    None) == inv
    assert lib.pa_decode_contiguous(16, 16, 16, 0, 128, None, None, 16, 1, 8, 2, 128, 0.1, 0, None, 0, 16, 1,
                                    None) == inv
    assert lib.pa_reshape_and_cache_slots(None, None, None, None, 1, None, None, 4, 100, None, 2, 128, 1,
                                          None) == inv
    assert lib.pa_reshape_and_cache_slots(None, None, None, None, 0, None, None, 4, 128, None, 2, 128, 1,
                                          None) == _lib.PA_OK
    # shared prefix: prefix not a multiple of the block size
    assert lib.pa_decode_shared_prefix(16, 16, 16, 16, 20, 16, 8, 16, 2, 8, 2, 128, 16, 64, 0.1, 0, 16, 1 << 20,
                                       16, 1, None, None) == inv


def test_sizes_past_the_int32_index_math_are_refused_on_the_host(lib):
    inv = _lib.PA_ERR_INVALID
    big = 2**31 - 1
    # a pool whose last row coordinate (one past it included) passes int32
    assert lib.pa_copy_blocks(16, 16, 16, 1, big, 16, 1, 64, 1, None) == inv
    assert lib.pa_copy_blocks(16, 16, 16, 1, big // 16, 16, 1, 64, 1, None) == inv
    # merge rows (request x query x head) past int32
    assert lib.pa_lse_merge(16, 1 << 40, 16, 1 << 20, 4096, 128, 4, 16, 0, 16, 1, None) == inv
    assert lib.pa_lse_merge(16, 1 << 40, 16, 65536, 32768, 128, 4, 16, 0, 16, 1, None) == inv   # 2^31 rows
    assert lib.pa_lse_merge(16, 1 << 40, 16, 65535, 32768, 128, 4, 16, 0, 16, 1, None) == _lib.PA_OK  # fits; one partition: nothing to merge
    # a workspace size query whose request x query count passes int32 is 0 (invalid)
    assert lib.pa_verify_workspace_size(1 << 30, 8, 8, 128, 64, 16, 128) == 0
    # a shared prefix against a table whose token capacity passes int32
    assert lib.pa_decode_shared_prefix(16, 16, 16, 16, 1024, 16, big, 16, 2, 8, 2, 128, 16, 64, 0.1, 0, 16,
                                       1 << 20, 16, 1, None, None) == inv
