"""The N>1 replica path of bench.py on CPU: two gloo ranks, the slowest
rank's time and the whole-job throughput (weak scaling, no data exchange)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    # rank r took (r + 1) * 10 ms for its K steps; the job takes the slowest
    ms = bench.reduce_max((rank + 1) * 10.0, ws, torch.device("cpu"))
    value = bench.whole_job_gbs(6e8, 100, ms * 1e-3, ws)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, value))


@pytest.mark.parametrize("ws", [2])
def test_two_replicas_report_the_max_time_and_the_summed_bytes(ws):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [20.0, 20.0]
    # 2 ranks x 600 MB x 100 steps over 20 ms
    assert all(abs(g[2] - 2 * 6e8 * 100 / 0.02 / 1e9) < 1e-6 for g in got)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_gbs(1e9, 10, 2.0, 1) == 5.0
