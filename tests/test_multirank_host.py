"""The benchmark's multi-GPU path on CPU: one process per rank over gloo, world size 2.
Each rank runs its own replica of the block (no data-path collective); the job's step
time is the maximum over ranks and the job throughput counts every rank's work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [40.0, 55.0][rank]
    ms = bench.reduce_max_ms(local_ms, world, dist)
    tf = bench.job_tflops(1e12, world, ms)
    out.put((rank, ms, tf))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_uses_the_slowest_rank():
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
    for rank, ms, tf in res:
        assert ms == 55.0
        assert tf == pytest.approx(2 * 1e12 / 0.055 / 1e12)
