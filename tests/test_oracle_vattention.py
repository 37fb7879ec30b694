"""The vAttention-style manager oracle ("vAttention 完全拆解"), pinned by the
page's formulas and numbers (golden `kv_sizing.json`) and its figure 2
walk-through of two request slots."""
import json
import os
import random

import numpy as np
import pytest

from oracle.vattention import NoPages, VAttnError, VirtualKV, pages_for, slot_row, tail_commit_bytes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_sizing.json")
MiB = 1 << 20


def test_slot_row_is_numpys_row_of_the_contiguous_layout():
    """Brute force: a [slots][max_len][H][D] array, flattened to token rows by
    numpy, holds token t of slot s at row slot_row(s, t, max_len)."""
    S, L, H, D = 3, 7, 2, 4
    a = np.arange(S * L * H * D).reshape(S, L, H, D)
    rows = a.reshape(S * L, H, D)
    for s in range(S):
        for t in range(L):
            assert np.array_equal(rows[slot_row(s, t, L)], a[s, t])


def test_slot_row_lands_on_the_pages_offset_of_the_request_slot():
    """"vAttention 完全拆解", core abstraction: slot reqId of a [B][L][H][D]
    tensor starts at byte offset(reqId) = reqId * L * H * D * P.  Numpy's
    row-major index of (reqId, t, 0, 0) in the Yi-34B worker's shape (golden
    fixture: L = 200000, H = 4, D = 128, P = 2), times P, must equal the
    page's offset plus t rows, and the row slot_row gives times the row size."""
    g = json.load(open(GOLDEN))["per_layer_k_or_v_slot"]
    L, H, D, P = g["length"], g["kv_heads"], g["head_dim"], g["elem_bytes"]
    B = 500
    for req, t in [(0, 0), (1, 0), (3, 5), (499, 199999), (250, 123456)]:
        byte = int(np.ravel_multi_index((req, t, 0, 0), (B, L, H, D))) * P
        assert byte == req * L * H * D * P + t * H * D * P       # the page's offset(reqId), then t rows
        assert slot_row(req, t, L) * H * D * P == byte
    assert L * H * D * P == g["exact_bytes"]                     # one slot = the printed ~200 MB


def test_pages_for_is_the_page_formula_with_whole_tiles():
    h = 4 * 128 * 2                                   # H=4, D=128, P=2 (the Yi-34B worker)
    # n_page = ceil(q H D P / G); with tile 1 exactly the printed formula
    assert pages_for(1000, h, 2 * MiB, tile=1) == 1
    assert pages_for(2048, h, 2 * MiB, tile=1) == 1   # 2 MiB exactly
    assert pages_for(2049, h, 2 * MiB, tile=1) == 2
    assert pages_for(5000, h, 2 * MiB, tile=1) == 3
    assert pages_for(0, h, 2 * MiB) == 0
    # with 16-token tiles the covered length is rounded up first
    assert pages_for(2040, h, 2 * MiB) == 1 and pages_for(2041, h, 2 * MiB) == 1
    assert pages_for(2049, h, 2 * MiB) == 2


def test_reservation_and_tail_commit_match_the_printed_numbers():
    g = json.load(open(GOLDEN))
    s = g["per_layer_k_or_v_slot"]
    v = VirtualKV(num_slots=g["virtual_reservation"]["batch"], max_len=s["length"],
                  layers=g["virtual_reservation"]["layers"], kv_heads=s["kv_heads"], head_dim=s["head_dim"],
                  elem_bytes=s["elem_bytes"], page_bytes=2 * MiB, max_pages=10 ** 6)
    assert v.virtual_offset(1) == s["exact_bytes"]          # offset(reqId) = reqId * L H D P
    assert v.virtual_offset(499) == 499 * s["exact_bytes"]
    # the page rounds S to 200 MB before multiplying: B * 200 MB = 100 GB (exactly 102.4 GB)
    assert v.B * 200e6 / 1e9 == g["virtual_reservation"]["printed_per_layer_tensor_gb"]
    assert abs(v.B * v.L * v.h / 1e9 / g["virtual_reservation"]["printed_per_layer_tensor_gb"] - 1) < 0.03
    assert round(v.B * v.L * v.h * v.tensors / 1e12) == g["virtual_reservation"]["printed_total_tb"]
    # W_max = 2 N' G: crossing one page boundary maps one page in each of the 2N' sub-tensors
    t = g["tail_commit"]
    assert tail_commit_bytes(t["layers"], t["page_mb"] * MiB) == t["printed_mb"] * MiB
    r = v.alloc_slot()
    lens = [0] * v.B
    per_page = 2 * MiB // v.h
    lens[r] = per_page
    v.step(lens)
    before = v.committed_bytes()
    lens[r] = per_page + 1
    v.step(lens)
    assert v.committed_bytes() - before == tail_commit_bytes(t["layers"], 2 * MiB)


def test_figure_two_walkthrough():
    """Two slots of one K tensor: (a) nothing mapped, (b) R1 maps its first
    page, (c) R1 grows to two pages and R2 gets one, (d) R1 finishes and keeps
    its pages, (e) R3 takes R1's id and reuses the mapped pages."""
    h = 1024
    per_page = 64 * 1024 // h                              # 64 tokens per 64 KB page
    v = VirtualKV(num_slots=2, max_len=4 * per_page, layers=1, kv_heads=1, head_dim=512, elem_bytes=2,
                  page_bytes=64 * 1024, max_pages=100)
    assert v.pages_in_use() == 0                           # (a)
    r1 = v.alloc_slot()
    v.step([10, 0] if r1 == 0 else [0, 10])
    assert v.mapped[r1] == 1                               # (b)
    r2 = v.alloc_slot()
    lens = [0, 0]
    lens[r1], lens[r2] = per_page + 5, 3
    v.step(lens)
    assert v.mapped[r1] == 2 and v.mapped[r2] == 1         # (c)
    v.free_slot(r1)
    lens[r1] = 0
    calls = v.map_calls
    v.step(lens)
    assert v.mapped[r1] == 2 and v.map_calls == calls      # (d) pages stay
    r3 = v.alloc_slot()
    assert r3 == r1                                        # (e) R3 takes R1's reqId ...
    lens[r3] = per_page + 40
    v.step(lens)
    assert v.map_calls == calls and v.mapped[r3] == 2      # ... and its mapped pages
    # R3 reads its token 5 from the row the page's offset(reqId) puts it at
    assert slot_row(r3, 5, v.L) * h == r3 * v.L * 1 * 512 * 2 + 5 * 1 * 512 * 2   # offset(reqId) + 5 rows


def test_shortage_is_all_or_nothing_and_reclaims_inactive_slots_first():
    v = VirtualKV(num_slots=4, max_len=1024, layers=1, kv_heads=1, head_dim=64, elem_bytes=2,
                  page_bytes=4096, max_pages=12)           # 32 tokens per page, 2 sub-tensors
    a, b = v.alloc_slot(), v.alloc_slot()
    lens = [0] * 4
    lens[a], lens[b] = 64, 64                              # 2 pages each x 2 tensors = 8
    v.step(lens)
    assert v.pool_free() == 4
    lens[a] = 160                                          # 5 pages: +3 x 2 = 6 > 4 free
    snap = (list(v.mapped), v.map_calls, v.unmap_calls)
    with pytest.raises(NoPages):
        v.step(lens)
    assert (list(v.mapped), v.map_calls, v.unmap_calls) == snap
    v.free_slot(b)                                         # b keeps 4 pages, reclaimable
    lens[b] = 0
    v.step(lens)
    assert v.mapped[a] == 5 and v.mapped[b] == 0 and v.unmap_calls == 4
    with pytest.raises(VAttnError):
        v.step([2000, 0, 0, 0])                            # past the reservation
    with pytest.raises(VAttnError):
        v.step([0, 0, 5, 0])                               # an inactive slot


def test_mapped_tokens_always_cover_whole_tiles_of_the_length():
    rng = random.Random(3)
    for _ in range(200):
        hb = rng.choice([64, 128, 384, 1024, 2048])
        G = rng.choice([4096, 65536, 2 * MiB])
        L = rng.choice([256, 1024, 4096])
        v = VirtualKV(2, L, 1, 1, hb // 2, 2, G, 10 ** 6)
        s = v.alloc_slot()
        n = rng.randrange(1, L + 1)
        lens = [0, 0]
        lens[s] = n
        v.step(lens)
        assert v.mapped_tokens(s) >= -(-n // 16) * 16 or v.mapped_tokens(s) == L
        assert v.mapped_tokens(s) % 16 == 0 or v.mapped_tokens(s) == L
