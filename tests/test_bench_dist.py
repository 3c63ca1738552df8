"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): the
timing crosses ranks only through a max-reduction and barriers; the whole-job
value counts every rank's FLOPs against the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t = 1.5 if rank == 0 else 2.5                  # rank 1 is the slowest
        m = bench.max_over_ranks(t)
        v = bench.aggregate_value(1e12, steps=10, world=world, max_seconds=m)
        r, w, lr = bench.dist_env()
        results[rank] = (m, v, r, w, lr)
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        for rank in range(world):
            m, v, r, w, lr = results[rank]
            assert m == 2.5                            # max over ranks
            assert v == pytest.approx(1e12 * 10 * 2 / 2.5 / 1e12)
            assert (r, w, lr) == (rank, world, rank)


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.aggregate_value(2e12, 5, 1, 2.0) == pytest.approx(5.0)
