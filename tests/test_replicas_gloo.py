"""The N > 1 path of bench.py on CPU: two ranks over gloo (world size 2, 127.0.0.1).

bench.py runs N independent replicas (the operation has no exchange step); ranks
meet only at a barrier and at the aggregation of the timed region: whole-job
units are summed over ranks and the time is the maximum over ranks. Rank 1's
reference arm returns without work and prints nothing.
"""
from __future__ import annotations

import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": "2",
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    try:
        ws, r, local = bench.dist_env()
        dist = bench.dist_init(ws, "gloo")
        dist.barrier()
        # rank r processed r + 1 units in 0.5 + r seconds
        units, sec = bench.aggregate(dist, float(r + 1), 0.5 + r)
        ref = bench.run_reference(None, ws, r) if r == 1 else "skipped"
        dist.barrier()
        dist.destroy_process_group()
        q.put((r, ws, local, units, sec, ref))
    except Exception as e:  # reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_ranks_sum_units_and_max_time():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r[0]: r for r in results}
    assert set(by_rank) == {0, 1}, results
    for r in (0, 1):
        rank, ws, local, units, sec, ref = by_rank[r]
        assert ws == 2 and local == r
        assert units == pytest.approx(3.0)      # 1 + 2 units
        assert sec == pytest.approx(1.5)        # max(0.5, 1.5) seconds
    assert by_rank[1][5] is None                # rank 1's reference arm: no work
