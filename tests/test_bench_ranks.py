"""The multi-process side of bench.py on CPU: two gloo ranks on 127.0.0.1 check the timing
collectives (max and sum over ranks), the whole-job value (units of every rank over the slowest
rank's time) and that only rank 0 of the reference arm does work. The path itself needs no
collective (replicas only); these are the bench's only cross-rank steps."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.rank_info()
        elapsed = 1.0 + rank  # rank 1 is the slow one
        emax = bench.rank_reduce(elapsed, "max", torch.device("cpu"))
        esum = bench.rank_reduce(elapsed, "sum", torch.device("cpu"))
        value = bench.whole_job_value(100, emax, w)

        class Args:  # the reference arm on a rank other than 0 must return at once
            steps, warmup = 10 ** 9, 10 ** 9
        t = None
        if rank != 0:
            import time
            t0 = time.perf_counter()
            bench.run_reference(Args, rank, w)
            t = time.perf_counter() - t0
        q.put((r, lr, w, emax, esum, value, t))
    finally:
        dist.destroy_process_group()


def test_bench_rank_aggregation_two_gloo_ranks():
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
    for rank, (r, lr, w, emax, esum, value, t) in enumerate(out):
        assert (r, lr, w) == (rank, rank, 2)
        assert emax == 2.0 and esum == 3.0
        assert value == pytest.approx(2 * 100 / 2.0)
    assert out[1][6] is not None and out[1][6] < 5.0


def test_single_rank_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.rank_reduce(3.5, "max", torch.device("cpu")) == 3.5
    assert bench.whole_job_value(10, 2.0, 1) == 5.0
