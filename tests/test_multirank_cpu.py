"""The benchmark's multi-rank path on CPU: two gloo ranks, each timing its own
independent block; the job time is the slowest rank's and the job value
counts every rank's work.  No GPU and no data-path collective."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_setup(world, backend="gloo")
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # rank r took (r + 1) * 100 ms over 4 steps for a 10 TFLOP block
    ms, tflops = bench.job_value(w, (r + 1) * 100.0, 4, 10e12)
    out[rank] = (ms, tflops)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # slowest rank: 200 ms over 4 steps = 50 ms per step; 2 blocks of 10 TFLOP per step
    for r in range(world):
        ms, tflops = res[r]
        assert ms == pytest.approx(50.0)
        assert tflops == pytest.approx(2 * 10e12 / 0.050 / 1e12)
