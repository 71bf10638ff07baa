"""The multi-process path of bench.py on CPU: two gloo ranks run the timing helpers
(barrier, max over ranks, sum of units) exactly as a torchrun launch would."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist(world)
    d.barrier()
    mx = d.max(float(rank + 1) * 1.5)            # e.g. per-rank ms per step
    sm = d.sum(float(64 * (rank + 1)))           # per-rank units
    d.barrier()
    q.put((rank, d.world, mx, sm))
    d.pg.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, mx, sm in res:
        assert w == world
        assert mx == pytest.approx(3.0)          # max over ranks
        assert sm == pytest.approx(192.0)        # units summed over ranks


def test_single_process_dist_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    d = bench.Dist(1)
    assert d.world == 1 and d.max(2.5) == 2.5 and d.sum(7.0) == 7.0
