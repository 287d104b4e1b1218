"""The benchmark's multi-process host logic on CPU: two ranks over gloo set up
the process group from the torchrun environment, meet at the barrier, and
both receive the largest elapsed time of all ranks (replicas, max over
ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank), "CUDA_VISIBLE_DEVICES": ""})
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(1.5 * (rank + 1), w)
    bench.barrier(w)
    q.put((rank, got, dist.get_backend()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(v == 3.0 for _, v, _ in res)
    assert all(b == "gloo" for _, _, b in res)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)
