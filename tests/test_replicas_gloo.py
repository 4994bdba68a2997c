"""Host logic of the multi-GPU bench run (replicas, weak scaling) with two
gloo ranks on CPU: the job's time is the slowest rank's, the job's throughput
counts every replica's parameters, and the reference arm runs on rank 0
only."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [12.5, 20.0][rank]
        worst = bench.max_over_ranks(ms, world, "cpu")
        thr = bench.job_throughput(1000, world, 4, worst)

        class A:
            workload, steps, warmup = "single", 1, 0
        ref = bench.run_reference(A, rank) if rank != 0 else "rank0"
        out.put((rank, worst, thr, ref))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, worst, thr, ref in res:
        assert worst == 20.0
        # 2 replicas x 1000 parameters x 4 steps in 20 ms
        assert thr == pytest.approx(2 * 1000 * 4 / 0.020)
    assert res[1][3] is None        # non-zero ranks print nothing
