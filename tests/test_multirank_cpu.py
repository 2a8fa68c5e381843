"""The multi-rank bench path on CPU: two gloo ranks, each timing its own replica, agree on
the slowest rank's time (the job's time). No GPU, no data-path collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        dist.barrier()
        local_ms = 10.0 + 5.0 * rank  # rank 1 is slower
        q.put((r, ws, local, bench.max_over_ranks(local_ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[3] == pytest.approx(15.0) for g in got)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
