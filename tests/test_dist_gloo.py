"""The multi-replica reduction of bench.py on two CPU ranks (gloo).

Each GPU runs an independent replica of the layer; the only cross-rank
step is the max-over-ranks of the step time that decides the whole-job
throughput.  This runs it on world_size 2 with the gloo backend.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.5][rank]
    slow = bench.max_over_ranks(ms, "cpu")
    v = bench.whole_job_value(1e12, world, slow)
    q.put((rank, slow, v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, v in out:
        assert slow == 5.5
        assert v == pytest.approx(2 * 1e12 / 5.5e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(4.25, "cpu") == 4.25
