"""Host side of the benchmark (CPU).

* The bench's algorithmic byte counts (the numerator of every roofline
  fraction it reports) equal the oracle's ``sizing`` counts, which are pinned
  by a brute-force count of touched elements, on the measured workloads'
  own tables.
* The reference arm (the float64 oracle) runs on the host without loading
  the CUDA library.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import workloads as W
from oracle import sizing

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", ["llama8b_gqa_decode", "prefix_shared_cow_decode", "spec_verify_decode",
                                  "tiny_paged_decode"])
def test_step_bytes_equal_the_oracle_sizing(name):
    wl = W.WORKLOADS[name]()
    hs = bench.HostStep(wl, value_seed=0)
    nb = bench.step_bytes(wl, hs.dec_lens, hs.dec_tables_np, None, None, len(hs.slots), 0)
    e = 2 if wl.dtype in ("bf16", "fp16") else None
    args = (wl.q_heads, wl.kv_heads, wl.head_dim, wl.block_size, e, wl.q_len)
    assert nb["decode"] == sizing.decode_step_bytes(hs.dec_lens, *args)
    tables = [hs.dec_tables_np[r] for r in range(len(hs.dec_lens))]
    assert nb["decode_unique"] == sizing.unique_kv_bytes(tables, hs.dec_lens, *args)
    if name == "prefix_shared_cow_decode":
        # the 2048-token prefix is read once: unique well below logical
        assert nb["decode_unique"] < nb["decode"] / 5
    else:
        assert nb["decode_unique"] == nb["decode"]


def test_host_step_tables_are_the_oracle_allocators():
    wl = W.WORKLOADS["llama8b_gqa_decode"]()
    hs = bench.HostStep(wl, value_seed=0)
    assert list(hs.dec_lens) == list(wl.decode_lens)
    bs = wl.block_size
    for r, L in enumerate(hs.dec_lens):
        n = -(-int(L) // bs)
        row = hs.dec_tables_np[r]
        assert (row[:n] >= 0).all() and (row[n:] == -1).all()
    used = np.concatenate([hs.dec_tables_np[r][:-(-int(L) // bs)] for r, L in enumerate(hs.dec_lens)])
    assert len(set(used.tolist())) == len(used)  # no block shared in this workload
    # the step's new token of every request lands in its last logical position
    for r, L in enumerate(hs.dec_lens):
        s = int(hs.slots[r])
        assert s // bs == hs.dec_tables_np[r][(int(L) - 1) // bs] and s % bs == (int(L) - 1) % bs


def test_reference_arm_runs_on_the_host_without_the_cuda_library():
    code = (
        "import runpy, sys\n"
        "sys.argv = ['bench.py', '--impl', 'reference', '--steps', '2', '--warmup', '3',"
        " '--workload', 'tiny_paged_decode']\n"
        "runpy.run_path('bench.py', run_name='__main__')\n"
        "maps = open('/proc/self/maps').read()\n"
        "assert 'libpa.so' not in maps, 'the reference arm loaded the CUDA library'\n"
        "assert 'paged_kv_cache_76_gb300' not in sys.modules\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["config"]["workload"] == "tiny_paged_decode"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
