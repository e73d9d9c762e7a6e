"""Multi-process host logic of the bench on CPU (gloo, world size 2).

The decode path shards as independent replicas: every rank runs the same step on its own
GPU and the job reports the slowest rank's time.  These tests cover that host logic -- the
barrier, the max over ranks, and the reference arm running on rank 0 only -- without a GPU.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    d = bench.Dist("gloo")
    d.barrier()
    m = d.max(float(rank + 1) * 1.5)
    d.barrier()
    ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})()) if rank == 1 else "skip"
    out.put((rank, m, ref))
    d.close()


def test_two_gloo_ranks_max_and_reference_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, m, ref = q.get(timeout=300)
        res[r] = (m, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == 3.0 and res[1][0] == 3.0   # max over ranks
    assert res[1][1] is None                         # the reference arm runs on rank 0 only
