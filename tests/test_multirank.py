"""The bench's multi-rank host logic (barrier, max over ranks, weak-scaling
aggregation) on world_size 2 with the gloo backend, on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), MXQ_BENCH_BACKEND="gloo")
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_init()
    bench.barrier(w)
    elapsed = bench.max_over_ranks(1.0 + 0.5 * r, w)          # rank 1 is the slow one
    value = w * bench.STEP_FLOP * 10 / elapsed / 1e12         # units of all ranks / max time
    q.put((r, w, elapsed, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == pytest.approx(1.5) for r in res)
    import bench
    assert res[0][3] == pytest.approx(2 * bench.STEP_FLOP * 10 / 1.5 / 1e12)
