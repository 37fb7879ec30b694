"""The C++ vAttention-style manager (pa_vkv_*, dry-run bookkeeping: no GPU)
against the oracle model, bit-exact after every operation."""
import numpy as np
import pytest

from oracle.vattention import NoPages as ONoPages
from oracle.vattention import VAttnError, VirtualKV as OVirtualKV
from paged_kv_cache_76_gb300 import _lib


@pytest.fixture(scope="module", autouse=True)
def built():
    try:
        _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()


def _c(*a, **k):
    from paged_kv_cache_76_gb300.vattention import VirtualKV
    return VirtualKV(*a, dry_run=True, **k)


def _do(target, op, *args):
    from paged_kv_cache_76_gb300.vattention import NoPages
    try:
        return ("ok", getattr(target, op)(*args))
    except (NoPages, ONoPages):
        return ("nopages", None)
    except (VAttnError, _lib.PAError):
        return ("err", None)


def _same(c, o):
    assert [c.slot_pages(s) for s in range(o.B)] == o.mapped
    st = c.stats()
    assert st["pages_mapped"] == o.pages_in_use() and st["map_calls"] == o.map_calls
    assert st["unmap_calls"] == o.unmap_calls and st["bytes_committed"] == o.committed_bytes()
    assert st["slot_pages"] == o.slot_pages
    tok = c.slot_tokens()
    assert [min(t // 16 * 16, o.L) for t in tok] == [o.mapped_tokens(s) for s in range(o.B)]


@pytest.mark.parametrize("seed", range(8))
def test_random_scripts_match_the_oracle(seed):
    rng = np.random.default_rng(500 + seed)
    B = int(rng.integers(1, 9))
    layers = int(rng.integers(1, 4))
    hkv, d = int(rng.choice([1, 2, 8])), int(rng.choice([64, 128]))
    row = hkv * d * 2
    page = int(rng.choice([4096, 16384, 65536]))
    # max_len: a multiple of 16 whose slot is a whole number of pages
    unit = np.lcm(16, page // np.gcd(page, row))
    L = int(unit * rng.integers(1, 4))
    budget = int(rng.integers(0, 2 * layers * B * (L * row // page) + 3))
    c = _c(B, L, layers, hkv, d, page_bytes=page, max_pages=budget)
    o = OVirtualKV(B, L, layers, hkv, d, 2, page, budget)
    lens = [0] * B
    refused = 0
    for step in range(300):
        kind = rng.choice(["alloc", "free", "step", "step", "step", "bad"])
        if kind == "alloc":
            rc, ro = _do(c, "alloc_slot"), _do(o, "alloc_slot")
            assert rc == ro, (step, rc, ro)
        elif kind == "free":
            s = int(rng.integers(0, B))
            rc, ro = _do(c, "free_slot", s), _do(o, "free_slot", s)
            assert rc[0] == ro[0]
            if rc[0] == "ok":
                lens[s] = 0
                # a freed slot's tokens stop counting at once, before the next step
                assert c.stats()["bytes_used"] == sum(lens) * row * 2 * layers
        elif kind == "step":
            new = list(lens)
            for s in range(B):
                if o.active[s]:
                    new[s] = int(min(L, max(0, new[s] + rng.integers(-8, 3 * unit // 2 + 1))))
            rc, ro = _do(c, "step", np.array(new)), _do(o, "step", new)
            assert rc[0] == ro[0], (step, rc, ro)
            if rc[0] == "ok":
                lens = new
                # the monitoring counters: bytes the tokens hold, refused steps
                assert c.stats()["bytes_used"] == sum(lens) * row * 2 * layers
            elif rc[0] == "nopages":
                refused += 1
            assert c.stats()["step_failures"] == refused
        else:  # a length past the reservation, or on an inactive slot
            bad = [0] * B
            bad[int(rng.integers(0, B))] = L + 16
            assert _do(c, "step", np.array(bad))[0] == _do(o, "step", bad)[0] == "err"
            idle = [s for s in range(B) if not o.active[s]]
            if idle:
                bad = list(lens)
                bad[idle[0]] = 16
                assert _do(c, "step", np.array(bad))[0] == _do(o, "step", bad)[0] == "err"
            assert c.stats()["bytes_used"] == sum(lens) * row * 2 * layers
        _same(c, o)


def test_creation_checks_alignment_and_sizes():
    from paged_kv_cache_76_gb300.vattention import VirtualKV
    with pytest.raises(_lib.PAError):
        VirtualKV(4, 100, 1, 8, 128, page_bytes=2 << 20, dry_run=True)        # max_len not a multiple of 16
    with pytest.raises(_lib.PAError):
        VirtualKV(4, 1008, 1, 8, 128, page_bytes=2 << 20, dry_run=True)       # slot not a whole number of pages
    with pytest.raises(_lib.PAError):
        VirtualKV(4, 1024, 1, 8, 128, page_bytes=0, dry_run=True)             # dry run needs the page size
    v = VirtualKV(4, 1024, 2, 8, 128, page_bytes=2 << 20, dry_run=True)
    assert v.stats()["slot_pages"] == 1 and v.stats()["bytes_reserved"] == 4 * 4 * 1024 * 2048
