"""The multi-GPU form of the benchmark is replicas only (every rank runs the
whole path on its own batch; no collective inside the path).  Its host
logic (barrier, the slowest rank's time, the whole-job value) runs here on
two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, loc = bench._dist()
        assert (r, w, loc) == (rank, world, rank)
        bench._barrier(w)
        step = bench._max_over_ranks(times[rank], w)
        out[rank] = (step, bench._job_value(1_000_000_000, step, w))
        bench._barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, times = 2, [0.5, 0.8]
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        step, value = out[r]
        assert step == pytest.approx(0.8)                 # both ranks see the slowest step
        assert value == pytest.approx(2 * 1.0 / 0.8e-3)  # GB/s: 2 ranks x 1 GB per 0.8 ms
