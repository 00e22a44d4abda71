"""The bench's multi-rank bookkeeping on CPU: two gloo ranks (world size 2)
exchange their timed regions; every rank must see the slowest one, and the
whole-job value counts all ranks' work in that time.  This is the path
`bench.py --gpus N` takes under torchrun, minus the GPU solves."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        slowest = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
        q.put((rank, r, w, local, slowest, bench.whole_job_value(w, 5, 1e6, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, (r, rr, w, local, slowest, value) in enumerate(got):
        assert (r, rr, w, local) == (rank, rank, 2, rank)
        assert slowest == 20.0                       # the slower rank's time
        assert value == 2 * 5 * 1e6 / 20.0           # both replicas' work in that time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(None, 3.5, None) == 3.5
    assert bench.whole_job_value(1, 4, 2.0, 8.0) == 1.0
