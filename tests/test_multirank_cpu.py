"""The multi-rank bench logic on CPU: two gloo ranks (127.0.0.1).

The path shards by independent token batches, so ranks exchange nothing but
a barrier and the max of their step times; the job's value is world x the
per-step work over the slowest rank's time (weak scaling)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank            # rank 1 is slower
    dist.barrier()
    worst = bench.max_over_ranks(ms, dist, "cpu")
    value = bench.whole_job_tflops(world, 1e12, worst)
    # the reference arm runs on rank 0 only; other ranks return at once
    class A:
        steps, warmup, gpus = 3, 3, world
    rc = bench.run_reference(A()) if rank == 1 else 0
    q.put((rank, worst, value, rc))
    dist.destroy_process_group()


def test_two_gloo_ranks():
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
    for rank, worst, value, rc in res:
        assert worst == 2.0                      # max over ranks
        assert abs(value - 2 * 1e12 / 2e-3 / 1e12) < 1e-9   # world * flops / slowest time
        assert rc == 0
