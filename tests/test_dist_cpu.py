"""The bench's multi-rank path on CPU: two processes over gloo (127.0.0.1)
run bench.dist_setup, bench.barrier and bench.max_over_ranks, the pieces a
multi-GPU run uses around its timed region (replicas only: no collective
touches the data path)."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        import torch.distributed as dist

        import bench
        w, r, _ = bench.dist_setup(world)
        bench.barrier(w)
        # the slowest rank's time is the job's time
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)
        bench.barrier(w)
        backend = dist.get_backend()
        dist.destroy_process_group()
        q.put((r, w, slowest, backend, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, world, None, None, repr(e)))


def test_max_over_ranks_two_gloo_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(q.get(timeout=180))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    errors = [e for (*_, e) in results if e]
    assert not errors, errors
    assert sorted(r for (r, *_) in results) == [0, 1]
    for (r, w, slowest, backend, _) in results:
        assert w == 2 and backend == "gloo"
        assert slowest == pytest.approx(15.0)
